"""Thin ctypes binding of the C-ABI in include/talker.h (argument marshalling only).

Every step of the forward runs in libtalker_gb300.so. PyTorch is used here only
to hold device memory and to name the CUDA stream. Loading fails loudly when the
library has not been built; there is no CPU fallback.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libtalker_gb300.so")

STATUS = {0: "TALKER_OK", 1: "TALKER_EINVAL", 2: "TALKER_EOVERFLOW", 3: "TALKER_ENOMEM", 4: "TALKER_ECUDA",
          5: "TALKER_ESTATE", 6: "TALKER_EDEVICE"}
DTYPE = {"f32": 0, "bf16": 1, "q8_0": 2}
LAYER_FIELDS = ("input_norm", "q_proj", "k_proj", "v_proj", "q_norm", "k_norm", "o_proj", "post_norm",
                "gate_proj", "up_proj", "down_proj")


class TalkerError(RuntimeError):
    def __init__(self, status, what):
        detail = ""
        if _lib is not None and status in (3, 4):
            detail = " (%s)" % _lib.talker_last_error().decode(errors="replace")
        super().__init__("%s failed: %s%s" % (what, STATUS.get(status, status), detail))
        self.status = status
        self.name = STATUS.get(status, str(status))


class Config(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int32), ("hidden", ctypes.c_int32), ("n_q_heads", ctypes.c_int32),
                ("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("intermediate", ctypes.c_int32),
                ("vocab", ctypes.c_int32), ("rms_eps", ctypes.c_float), ("rope_theta", ctypes.c_float),
                ("weight_dtype", ctypes.c_int32), ("kv_dtype", ctypes.c_int32)]


class LayerPtrs(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in LAYER_FIELDS]


class WeightPtrs(ctypes.Structure):
    _fields_ = [("layers", ctypes.POINTER(LayerPtrs)), ("final_norm", ctypes.c_void_p),
                ("codec_head", ctypes.c_void_p)]


_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libtalker_gb300.so and declare its prototypes. Raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError("CUDA library %s is missing: build it with `python -c 'import __graft_entry__ as g; "
                           "g.build()'` (there is no CPU fallback)" % path)
    lib = ctypes.CDLL(path)
    vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    st = ctypes.c_int
    proto = {
        "talker_create": (st, [ctypes.POINTER(Config), ctypes.POINTER(WeightPtrs), vp, ctypes.POINTER(vp)]),
        "talker_destroy": (None, [vp]),
        "talker_kv_init_batched": (st, [vp, ctypes.c_int, ctypes.c_int]),
        "talker_kv_rewind": (st, [vp, ctypes.c_int, ctypes.c_int]),
        "talker_cur_len": (st, [vp, ctypes.c_int, ctypes.POINTER(ctypes.c_int)]),
        "talker_prefill": (st, [vp, ctypes.c_int, vp, ctypes.c_int, vp, vp, vp]),
        "talker_prefill_append": (st, [vp, ctypes.c_int, vp, ctypes.c_int, vp, vp, vp]),
        "talker_frame": (st, [vp, vp, ctypes.c_int, ctypes.c_int, ctypes.POINTER(ctypes.c_int), ctypes.POINTER(vp),
                              vp, vp]),
        "talker_prefill_batched": (st, [vp, ctypes.c_int, vp, ctypes.c_int, vp, vp, vp]),
        "talker_set_logit_suppression": (st, [vp, ctypes.c_int, ctypes.c_int]),
        "talker_set_code_tables": (st, [vp, ctypes.POINTER(vp), ctypes.POINTER(ctypes.c_int), ctypes.c_int,
                                        ctypes.c_int]),
        "talker_decode_codes": (st, [vp, vp, vp, ctypes.c_int, vp, vp, vp]),
        "talker_decode": (st, [vp, vp, ctypes.c_int, vp, vp, vp]),
        "talker_prefill_all_rows": (st, [vp, ctypes.c_int, vp, ctypes.c_int, vp, vp]),
        "talker_kv_import": (st, [vp, ctypes.c_int, vp, vp, ctypes.c_int]),
        "talker_kv_export": (st, [vp, ctypes.c_int, vp, vp, ctypes.c_int]),
        "talker_sync_status": (st, [vp, ctypes.POINTER(i32)]),
        "talker_status_str": (ctypes.c_char_p, [st]),
        "talker_kernel_launches": (i64, [vp]),
        "talker_last_error": (ctypes.c_char_p, []),
        "talker_set_decode_mode": (st, [vp, ctypes.c_int]),
        "talker_set_prefill_mode": (st, [vp, ctypes.c_int]),
        "talker_head_argmax_noalloc": (st, [vp, ctypes.c_int, ctypes.c_int, vp, ctypes.c_int, ctypes.c_int, vp, vp,
                                            vp]),
        "talker_test_gemm_bf16": (st, [vp, ctypes.c_int, ctypes.c_int, vp, ctypes.c_int, vp, ctypes.c_int,
                                       ctypes.c_int, vp]),
        "talker_test_gemm_swiglu_bf16": (st, [vp, ctypes.c_int, ctypes.c_int, vp, ctypes.c_int, vp, vp]),
    }
    for name, (res, args) in proto.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def make_config(geom) -> Config:
    return Config(geom.n_layers, geom.hidden, geom.n_q_heads, geom.n_kv_heads, geom.head_dim, geom.intermediate,
                  geom.vocab, geom.rms_eps, geom.rope_theta, DTYPE[geom.weight_dtype], DTYPE[geom.kv_dtype])


def _ptr(t):
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


class Talker:
    """One library handle: weights, a paged KV cache and the decode graphs, on the current CUDA device."""

    def __init__(self, geom, weights: dict, stream=None):
        import torch
        self.torch = torch
        self.g = geom
        self.lib = load_library()
        self.dev = torch.device("cuda", torch.cuda.current_device())
        self.stream = stream if stream is not None else torch.cuda.current_stream(self.dev)
        wdt = torch.bfloat16 if geom.weight_dtype == "bf16" else torch.float32
        keep = []

        def up(a, dtype):
            t = torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(self.dev).to(dtype)
            keep.append(t)
            return t.data_ptr()

        layers = (LayerPtrs * geom.n_layers)()
        for l, lw in enumerate(weights["layers"]):
            for name in LAYER_FIELDS:
                is_norm = name.endswith("norm")
                setattr(layers[l], name, up(lw[name], torch.float32 if is_norm else wdt))
        wp = WeightPtrs(layers, up(weights["final_norm"], torch.float32), up(weights["codec_head"], wdt))
        cfg = make_config(geom)
        h = ctypes.c_void_p()
        self._check(self.lib.talker_create(ctypes.byref(cfg), ctypes.byref(wp),
                                           ctypes.c_void_p(self.stream.cuda_stream), ctypes.byref(h)),
                    "talker_create")
        self.h = h
        del keep  # the library copied the weights (talker_create synchronises its stream)

    @staticmethod
    def _check(status, what):
        if status != 0:
            raise TalkerError(status, what)

    def close(self):
        if getattr(self, "h", None):
            self.lib.talker_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # -- cache -------------------------------------------------------------------
    def kv_init_batched(self, n_streams: int, max_seq_len: int):
        self._check(self.lib.talker_kv_init_batched(self.h, n_streams, max_seq_len), "talker_kv_init_batched")

    def rewind(self, stream: int, new_len: int):
        self._check(self.lib.talker_kv_rewind(self.h, stream, new_len), "talker_kv_rewind")

    def cur_len(self, stream: int) -> int:
        out = ctypes.c_int()
        self._check(self.lib.talker_cur_len(self.h, stream, ctypes.byref(out)), "talker_cur_len")
        return out.value

    def kv_import(self, stream: int, k, v, length: int):
        self._check(self.lib.talker_kv_import(self.h, stream, _ptr(k), _ptr(v), length), "talker_kv_import")

    def kv_export(self, stream: int, k, v, length: int):
        self._check(self.lib.talker_kv_export(self.h, stream, _ptr(k), _ptr(v), length), "talker_kv_export")

    # -- forward -----------------------------------------------------------------
    def _out(self, *shape, dtype=None):
        return self.torch.empty(*shape, device=self.dev, dtype=dtype or self.torch.float32)

    def prefill(self, stream: int, emb, hidden=True, argmax=True):
        """emb: [T, H] f32 cuda. Returns (hidden_last [H] | None, logits_last [V], argmax [1] | None)."""
        T = emb.shape[0]
        lg = self._out(self.g.vocab)
        hd = self._out(self.g.hidden) if hidden else None
        am = self._out(1, dtype=self.torch.int32) if argmax else None
        self._check(self.lib.talker_prefill(self.h, stream, _ptr(emb), T, _ptr(hd), _ptr(lg), _ptr(am)),
                    "talker_prefill")
        return hd, lg, am

    def prefill_append(self, stream: int, emb, hidden=True, argmax=True):
        """Append emb [T, H] after the stream's cached rows (chunked prefill). Returns like prefill."""
        T = emb.shape[0]
        lg = self._out(self.g.vocab)
        hd = self._out(self.g.hidden) if hidden else None
        am = self._out(1, dtype=self.torch.int32) if argmax else None
        self._check(self.lib.talker_prefill_append(self.h, stream, _ptr(emb), T, _ptr(hd), _ptr(lg), _ptr(am)),
                    "talker_prefill_append")
        return hd, lg, am

    def prefill_batched(self, emb, hidden=True, argmax=True):
        """emb [B, T, H] f32 cuda: streams 0..B-1 prefilled with T rows each. Returns per-stream last rows."""
        B, T = emb.shape[0], emb.shape[1]
        lg = self._out(B, self.g.vocab)
        hd = self._out(B, self.g.hidden) if hidden else None
        am = self._out(B, dtype=self.torch.int32) if argmax else None
        self._check(self.lib.talker_prefill_batched(self.h, B, _ptr(emb), T, _ptr(hd), _ptr(lg), _ptr(am)),
                    "talker_prefill_batched")
        return hd, lg, am

    def prefill_all_rows(self, stream: int, emb, hidden=True):
        T = emb.shape[0]
        lg = self._out(T, self.g.vocab)
        hd = self._out(T, self.g.hidden) if hidden else None
        self._check(self.lib.talker_prefill_all_rows(self.h, stream, _ptr(emb), T, _ptr(hd), _ptr(lg)),
                    "talker_prefill_all_rows")
        return hd, lg

    def decode(self, emb, logits=None, hidden=None, argmax=None):
        """emb: [B, H] f32 cuda for streams 0..B-1. Outputs may be passed in to reuse the decode graph."""
        B = emb.shape[0]
        if logits is None:
            logits = self._out(B, self.g.vocab)
        self._check(self.lib.talker_decode(self.h, _ptr(emb), B, _ptr(logits), _ptr(hidden), _ptr(argmax)),
                    "talker_decode")
        return logits, hidden, argmax

    def set_logit_suppression(self, vocab_tail: int, eos_id: int):
        self._check(self.lib.talker_set_logit_suppression(self.h, vocab_tail, eos_id), "talker_set_logit_suppression")

    def set_code_tables(self, tables, dtype_bf16: bool):
        """tables: list of cuda tensors [V_g, H] (kept referenced by this object while registered)."""
        self._code_tables = list(tables)
        n = len(tables)
        arr = (ctypes.c_void_p * max(1, n))(*[t.data_ptr() for t in tables])
        voc = (ctypes.c_int * max(1, n))(*[int(t.shape[0]) for t in tables])
        self._check(self.lib.talker_set_code_tables(self.h, arr, voc, n, 1 if dtype_bf16 else 0),
                    "talker_set_code_tables")

    def decode_codes(self, ids, overlay=None, logits=None, hidden=None, argmax=None):
        """ids: int32 cuda [n_tables, B]; overlay: f32 cuda [B, H] or None."""
        B = ids.shape[1]
        if logits is None:
            logits = self._out(B, self.g.vocab)
        self._check(self.lib.talker_decode_codes(self.h, _ptr(ids), _ptr(overlay), B, _ptr(logits), _ptr(hidden),
                                                 _ptr(argmax)), "talker_decode_codes")
        return logits, hidden, argmax

    def frame(self, emb, table_of_step, codes, logits=None, heads=None):
        """emb [T0, H] f32 cuda; table_of_step: list of table indices (one per step); codes int32 cuda
        [n_steps + 1]; logits f32 cuda [n_steps + 1, V] or None; heads: None (codec_head for every
        code) or a list of n_steps + 1 cuda tensors [V, H] in the weight dtype (heads[0] for the
        prefill's code, heads[i + 1] for step i's)."""
        n = len(table_of_step)
        arr = (ctypes.c_int * max(1, n))(*table_of_step)
        hp = None
        if heads is not None:
            if len(heads) != n + 1:
                raise ValueError("frame: need n_steps + 1 heads")
            hp = (ctypes.c_void_p * (n + 1))(*[h.data_ptr() for h in heads])
        self._check(self.lib.talker_frame(self.h, _ptr(emb), emb.shape[0], n, arr, hp, _ptr(codes), _ptr(logits)),
                    "talker_frame")

    def set_decode_mode(self, mode: int):
        """0 automatic, 2 the GEMV graph, 3 the tensor-core graph."""
        self._check(self.lib.talker_set_decode_mode(self.h, mode), "talker_set_decode_mode")

    def set_prefill_mode(self, mode: int):
        """0 automatic (tensor cores for bf16 weights and T >= 16), 2 GEMV kernels, 3 / 4 tensor
        cores with the mma.sync / tcgen05 prefill attention at any T."""
        self._check(self.lib.talker_set_prefill_mode(self.h, mode), "talker_set_prefill_mode")

    def sync_status(self) -> int:
        code = ctypes.c_int32(0)
        st = self.lib.talker_sync_status(self.h, ctypes.byref(code))
        if st not in (0, 6):
            raise TalkerError(st, "talker_sync_status")
        return code.value

    def kernel_launches(self) -> int:
        return int(self.lib.talker_kernel_launches(self.h))


def test_gemm_swiglu_bf16(A, B, out):
    """Test support: out[M, N/2] = bf16(silu(A @ B[0::2].T) * (A @ B[1::2].T)) on the tensor-core
    GEMM's SwiGLU epilogue (A [M,K], B [N,K] bf16 with gate/up rows interleaved; out bf16)."""
    import torch
    lib = load_library()
    M, K = A.shape
    N = B.shape[0]
    st = lib.talker_test_gemm_swiglu_bf16(_ptr(A), M, K, _ptr(B), N, _ptr(out),
                                          ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    if st != 0:
        raise TalkerError(st, "talker_test_gemm_swiglu_bf16")
    return out


def test_gemm_bf16(A, B, out, accumulate=False, splits=1):
    """Test support: out (+)= A @ B.T on the tensor-core GEMM (A [M,K], B [N,K] bf16; out f32 [M,N])."""
    import torch
    lib = load_library()
    M, K = A.shape
    N = B.shape[0]
    st = lib.talker_test_gemm_bf16(_ptr(A), M, K, _ptr(B), N, _ptr(out), int(accumulate), splits,
                                   ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    if st != 0:
        raise TalkerError(st, "talker_test_gemm_bf16")
    return out


def head_argmax_noalloc(hidden, W, logits, argmax, weight_dtype):
    """logits = hidden @ W.T and per-row argmax through the allocation-free entry point."""
    import torch
    lib = load_library()
    rows, H = hidden.shape
    st = lib.talker_head_argmax_noalloc(_ptr(hidden), rows, H, _ptr(W), W.shape[0], DTYPE[weight_dtype],
                                        _ptr(logits), _ptr(argmax),
                                        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    if st != 0:
        raise TalkerError(st, "talker_head_argmax_noalloc")
