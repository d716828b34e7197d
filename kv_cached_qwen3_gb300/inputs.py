"""Seeded synthetic inputs for the Talker decoder workloads.

This module only draws random numbers and arranges them into arrays: model
geometry, weights, embeddings, stream lengths and pre-filled KV contents. It
holds none of the forward arithmetic, so both the fp64 oracle and the CUDA
path can take their inputs from it without sharing any computation.

Distributions (the workloads of "qwentts.cpp/src/talker-forward.h" and the
rightkit-qts "tts_transformer.rs" page, TtsTransformerConfig defaults):
  * linear weights   ~ N(0, 0.02), stored [out, in] row-major;
  * norm gains       ~ 1 + N(0, 0.05), always fp32;
  * embeddings       ~ N(0, 1) fp32, [rows, hidden];
  * pre-filled K/V   ~ N(0, 1), standing in for post-QK-norm/RoPE keys.
Where the geometry is bf16, linear weights are drawn in fp64, cast to fp32 and
then rounded to bf16 (round-to-nearest-even); the returned fp32 arrays hold
those bf16 values exactly.

Every tensor is split into fixed chunks, and chunk c of tensor i is drawn from
``PCG64(SeedSequence([seed, i, c]))``. The values therefore do not depend on
the thread count or the machine, and generation runs on all host cores.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field, replace

import numpy as np

_CHUNK = 1 << 21          # elements per independently seeded chunk
_EMB_BLOCK = 64           # embedding rows per independently seeded block
_EMB_SEED_OFFSET = 1000   # embeddings come from an independent seed stream
_KV_SEED_OFFSET = 2000    # pre-filled KV contents likewise
_LEN_SEED_OFFSET = 3000   # per-stream start lengths likewise


@dataclass(frozen=True)
class Geometry:
    """Decoder geometry and storage formats (names as in TtsTransformerConfig)."""
    n_layers: int
    hidden: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    intermediate: int
    vocab: int
    rms_eps: float = 1e-6
    rope_theta: float = 1e6
    weight_dtype: str = "bf16"   # "f32" | "bf16" for the linear weights
    kv_dtype: str = "bf16"       # "f32" | "bf16" for the KV cache

    @property
    def q_dim(self) -> int:
        return self.n_q_heads * self.head_dim

    @property
    def kv_dim(self) -> int:
        return self.n_kv_heads * self.head_dim

    def n_linear_params(self) -> int:
        per_layer = (self.q_dim + 2 * self.kv_dim) * self.hidden + self.hidden * self.q_dim \
            + 2 * self.intermediate * self.hidden + self.hidden * self.intermediate
        return self.n_layers * per_layer + self.vocab * self.hidden


TINY = Geometry(n_layers=2, hidden=128, n_q_heads=4, n_kv_heads=2, head_dim=32,
                intermediate=384, vocab=256, weight_dtype="f32", kv_dtype="f32")
TALKER = Geometry(n_layers=28, hidden=1024, n_q_heads=16, n_kv_heads=8, head_dim=128,
                  intermediate=3072, vocab=3072)
PREDICTOR = replace(TALKER, n_layers=5, vocab=2048)


@dataclass(frozen=True)
class Workload:
    """One of the five synthetic workloads: geometry plus the sizes it runs at."""
    name: str
    geometry: Geometry
    seed: int
    prefill_T: int
    decode_steps: int
    n_streams: int = 1
    frames: int = 0                      # predictor loop: frames of (prefill + steps)
    start_len_range: tuple = ()          # batched: uniform start lengths (inclusive)
    long_lengths: tuple = ()             # long context: decode cache lengths
    extra: dict = field(default_factory=dict)


WORKLOADS = {
    "tiny": Workload("tiny", TINY, seed=0, prefill_T=16, decode_steps=16),
    "talker_b1": Workload("talker_b1", TALKER, seed=1, prefill_T=96, decode_steps=512),
    "predictor_loop": Workload("predictor_loop", PREDICTOR, seed=2, prefill_T=2, decode_steps=15,
                               frames=256),
    "batched16": Workload("batched16", TALKER, seed=3, prefill_T=0, decode_steps=256, n_streams=16,
                          start_len_range=(128, 2048)),
    "long_context": Workload("long_context", TALKER, seed=4, prefill_T=4096, decode_steps=1,
                             long_lengths=(8192, 16384, 32768)),
}

LINEAR_NAMES = ("q_proj", "k_proj", "v_proj", "o_proj", "gate_proj", "up_proj", "down_proj")
NORM_NAMES = ("input_norm", "q_norm", "k_norm", "post_norm")


def tensor_specs(g: Geometry):
    """(name, shape, kind) of every weight tensor, in the fixed draw order."""
    H, hd, I = g.hidden, g.head_dim, g.intermediate
    specs = []
    for l in range(g.n_layers):
        specs += [
            ((l, "input_norm"), (H,), "norm"),
            ((l, "q_proj"), (g.q_dim, H), "linear"),
            ((l, "k_proj"), (g.kv_dim, H), "linear"),
            ((l, "v_proj"), (g.kv_dim, H), "linear"),
            ((l, "q_norm"), (hd,), "norm"),
            ((l, "k_norm"), (hd,), "norm"),
            ((l, "o_proj"), (H, g.q_dim), "linear"),
            ((l, "post_norm"), (H,), "norm"),
            ((l, "gate_proj"), (I, H), "linear"),
            ((l, "up_proj"), (I, H), "linear"),
            ((l, "down_proj"), (H, I), "linear"),
        ]
    specs += [((None, "final_norm"), (H,), "norm"), ((None, "codec_head"), (g.vocab, H), "linear")]
    return specs


def _threads() -> int:
    return max(1, min(32, os.cpu_count() or 1))


def _normal_chunked(entropy: list, n: int, pool: ThreadPoolExecutor | None) -> np.ndarray:
    """n fp64 N(0,1) draws, chunk c from PCG64(SeedSequence(entropy + [c]))."""
    out = np.empty(n, np.float64)
    bounds = [(c, c * _CHUNK, min(n, (c + 1) * _CHUNK)) for c in range((n + _CHUNK - 1) // _CHUNK)]

    def fill(b):
        c, lo, hi = b
        rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence(entropy + [c])))
        out[lo:hi] = rng.standard_normal(hi - lo)

    if pool is None or len(bounds) == 1:
        for b in bounds:
            fill(b)
    else:
        list(pool.map(fill, bounds))
    return out


def round_to_bf16(a: np.ndarray) -> np.ndarray:
    """fp32 array -> fp32 array holding the bf16 round-to-nearest-even values."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a, np.float32))
    return t.to(torch.bfloat16).to(torch.float32).numpy()


def bf16_bits(a: np.ndarray) -> np.ndarray:
    """fp32 array of bf16-representable values -> uint16 bit patterns (exact)."""
    a = np.ascontiguousarray(a, np.float32)
    return (a.view(np.uint32) >> 16).astype(np.uint16)


def make_weights(g: Geometry, seed: int) -> dict:
    """Seeded weights: {"layers": [ {name: array} ], "final_norm": ..., "codec_head": ...}.

    Linear weights are fp32 arrays (bf16-valued when g.weight_dtype == "bf16");
    norm gains are fp32.
    """
    layers = [dict() for _ in range(g.n_layers)]
    out = {"layers": layers}
    with ThreadPoolExecutor(_threads()) as pool:
        for idx, ((l, name), shape, kind) in enumerate(tensor_specs(g)):
            n = int(np.prod(shape))
            z = _normal_chunked([seed, idx], n, pool)
            if kind == "linear":
                a = (z * 0.02).astype(np.float32).reshape(shape)
                if g.weight_dtype == "bf16":
                    a = round_to_bf16(a)
            else:
                a = (1.0 + 0.05 * z).astype(np.float32).reshape(shape)
            if l is None:
                out[name] = a
            else:
                layers[l][name] = a
    return out


def make_embeddings(g: Geometry, seed: int, row_begin: int, row_end: int, stream: int = 0) -> np.ndarray:
    """Rows [row_begin, row_end) of stream `stream`'s N(0,1) embedding sequence, fp32 [rows, hidden].

    Block b of 64 rows comes from PCG64(SeedSequence([seed + 1000, stream, b])), so a row's values do
    not depend on how many rows are requested.
    """
    H = g.hidden
    if row_end <= row_begin:
        return np.zeros((0, H), np.float32)
    b0, b1 = row_begin // _EMB_BLOCK, (row_end - 1) // _EMB_BLOCK
    blocks = []
    for b in range(b0, b1 + 1):
        rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed + _EMB_SEED_OFFSET, stream, b])))
        blocks.append(rng.standard_normal((_EMB_BLOCK, H)).astype(np.float32))
    allrows = np.concatenate(blocks, axis=0)
    off = row_begin - b0 * _EMB_BLOCK
    return np.ascontiguousarray(allrows[off:off + (row_end - row_begin)])


def make_start_lengths(seed: int, n_streams: int, lo: int, hi: int) -> np.ndarray:
    """Per-stream start lengths ~ U{lo..hi} (inclusive), int32."""
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed + _LEN_SEED_OFFSET])))
    return rng.integers(lo, hi + 1, size=n_streams).astype(np.int32)


def make_kv_layer(g: Geometry, seed: int, layer: int, length: int, stream: int = 0) -> tuple:
    """Pre-filled cache contents for one layer: K, V fp32 [n_kv_heads, length, head_dim] ~ N(0,1).

    Values are rounded to bf16 when g.kv_dtype == "bf16" (the cache then holds them exactly).
    Row p of a (layer, head) does not depend on `length`: the draws are laid out position-major
    in chunks, [pos][head][dim].
    """
    nkv, hd = g.n_kv_heads, g.head_dim
    n = length * nkv * hd
    res = [np.empty((nkv, length, hd), np.float32) for _ in range(2)]
    step = 512                                   # positions per conversion job
    with ThreadPoolExecutor(_threads()) as pool:
        zs = [_normal_chunked([seed + _KV_SEED_OFFSET, stream, layer, kind], n, pool) for kind in (0, 1)]

        def convert(job):
            kind, p0 = job
            p1 = min(length, p0 + step)
            src = zs[kind][p0 * nkv * hd:p1 * nkv * hd].reshape(p1 - p0, nkv, hd)
            res[kind][:, p0:p1, :] = src.transpose(1, 0, 2)

        list(pool.map(convert, [(kind, p0) for kind in (0, 1) for p0 in range(0, length, step)]))
    if g.kv_dtype == "bf16":
        res = [round_to_bf16(a) for a in res]
    return res[0], res[1]
