"""fp64 CPU oracle of the KV-cached Qwen3 "Talker" decoder forward.

TEST INFRASTRUCTURE. Only tests/, the smoke check in __graft_entry__ and the
CPU-baseline leg of bench.py may import this module. It shares no code with the
CUDA library and never calls it; the library never calls this.

Everything is computed in float64 from the stored weight values (fp32, or fp32
holding bf16 values, widened exactly). The forward follows these page sections:

  "qwentts.cpp/src/talker-forward.h"
    - talker_layer_forward: pre-norm RMSNorm and gain; bias-free Q/K/V
      projections; per-head QK-RMSNorm with an [hd] gain and the same eps;
      RoPE NEOX (rotate-half) with the mrope axes collapsed to one position;
      K/V written into the cache at the rows of the fresh positions; GQA
      scaled-dot-product attention with scale 1/sqrt(hd) over the causal
      window; o_proj and residual; post-attention RMSNorm; SwiGLU MLP
      (gate, up, down) and residual.
    - talker_forward_core: positions n_past..n_past+T-1, causal mask "key k
      visible to query q iff k <= n_past + q", final RMSNorm and codec_head,
      last-row readback, cur_len = n_past + T afterwards.
    - talker_forward_prefill: rewind the stream's cache to 0, T <= max_seq_len.
    - talker_forward_decode: one row per stream at position cur_len[s],
      window [0, cur_len[s]], overflow check cur_len+1 <= max_seq_len, then
      cur_len[s] += 1.
  "transcribe.cpp/src/causal_lm/causal_lm.cpp": Qwen3 block (bias-free
    projections, "NeoX rotate_half" RoPE, GQA by repeat_interleave of the KV
    heads, i.e. q head h reads KV head h // (n_q / n_kv)).
  rightkit-qts "tts_transformer.rs": the explicit SwiGLU form silu(gate) * up;
    the uncached "recompute" path that re-runs the full sequence (mode A here);
    the code predictor's frame (predict_remaining_codebooks_kv_with_cache), whose
    prefill projects with heads[0] and generation step g with heads[g], the
    step's input being the previous code's row of its embedding table.

Readings taken where the pages leave a step open (each is listed in the design
notes): RoPE angle for pair i at position p is p * theta**(-2 i / hd), pairing
element i with element i + hd/2, position = absolute cache row; eps sits inside
the square root and the norm gain multiplies directly (no "1 + w"); the mask is
additive 0 / -inf, i.e. a softmax over exactly the keys j <= p; silu(z) =
z / (1 + exp(-z)); "final hidden" is the output of the final norm; argmax ties
go to the lowest index.

Two modes that must agree:
  A  forward_full: the uncached full-sequence forward with an explicit T x T
     causal mask (no cache anywhere);
  B  OracleCache: the incremental cached forward (prefill / decode / rewind /
     import / export), mirroring the cache semantics of talker_forward_core
     and talker_forward_decode.

Parity of the end-to-end values against any external implementation is
unpinned (the pages publish no weights or worked numbers); each step is pinned
by the closed forms and invariants in tests/test_oracle_pins.py.
"""
from __future__ import annotations

import numpy as np

F64 = np.float64


# ----------------------------------------------------------------------------- steps

def rms_norm(x, w, eps):
    """x / sqrt(mean(x^2) + eps) * w over the last axis (talker_layer_forward, "Pre-norm")."""
    x = np.asarray(x, F64)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * np.asarray(w, F64)


def rope_neox(x, positions, theta):
    """NEOX rotate-half RoPE (talker_layer_forward, "RoPE NEOX (half-split)").

    x: [rows, heads, hd]; positions: [rows] absolute cache rows.
    Pair (x_i, x_{i+hd/2}) at angle phi = p * theta**(-2 i / hd) becomes
    (x_i cos phi - x_{i+hd/2} sin phi, x_{i+hd/2} cos phi + x_i sin phi).
    """
    x = np.asarray(x, F64)
    hd = x.shape[-1]
    half = hd // 2
    i = np.arange(half, dtype=F64)
    inv_freq = np.power(F64(theta), -2.0 * i / hd)
    phi = np.asarray(positions, F64)[:, None] * inv_freq[None, :]          # [rows, half]
    c = np.cos(phi)[:, None, :]
    s = np.sin(phi)[:, None, :]
    a, b = x[..., :half], x[..., half:]
    return np.concatenate([a * c - b * s, b * c + a * s], axis=-1)


def silu(z):
    """silu(z) = z / (1 + exp(-z)) (tts_transformer.rs, ggml_silu on the gate)."""
    z = np.asarray(z, F64)
    return z / (1.0 + np.exp(-z))


def softmax(s, axis=-1):
    """Max-subtracted softmax; -inf entries get probability 0."""
    m = np.max(s, axis=axis, keepdims=True)
    e = np.exp(s - m)
    return e / np.sum(e, axis=axis, keepdims=True)


def kv_group(h, n_q_heads, n_kv_heads):
    """KV head read by q head h: repeat_interleave of the KV heads (causal_lm.cpp, GQA)."""
    return h // (n_q_heads // n_kv_heads)


def attend_one(q, K, V, n_visible):
    """One query row against cached keys [0, n_visible) (talker_layer_forward, attention).

    q: [n_q, hd]; K, V: [n_kv, >= n_visible, hd]. Returns [n_q, hd].
    """
    n_q, hd = q.shape
    n_kv = K.shape[0]
    out = np.empty((n_q, hd), F64)
    for h in range(n_q):
        g = kv_group(h, n_q, n_kv)
        s = (K[g, :n_visible] @ q[h]) / np.sqrt(F64(hd))
        out[h] = softmax(s) @ V[g, :n_visible]
    return out


def argmax_low(v):
    """Index of the maximum, the lowest index on ties (np.argmax's rule)."""
    return int(np.argmax(np.asarray(v)))


# ----------------------------------------------------------------------------- model

class Oracle:
    """Weights widened to fp64 plus the per-layer pieces of the forward."""

    def __init__(self, geom, weights):
        self.g = geom
        self.layers = []
        for lw in weights["layers"]:
            self.layers.append({k: np.asarray(v, F64) for k, v in lw.items()})
        self.final_norm = np.asarray(weights["final_norm"], F64)
        self.codec_head = np.asarray(weights["codec_head"], F64)

    # -- pieces of talker_layer_forward --------------------------------------
    def qkv(self, l, x, positions):
        """Pre-norm, Q/K/V projections, per-head QK-norm, RoPE. Returns q [T,nq,hd], k, v [T,nkv,hd]."""
        g, w = self.g, self.layers[l]
        T = x.shape[0]
        h = rms_norm(x, w["input_norm"], g.rms_eps)
        q = (h @ w["q_proj"].T).reshape(T, g.n_q_heads, g.head_dim)
        k = (h @ w["k_proj"].T).reshape(T, g.n_kv_heads, g.head_dim)
        v = (h @ w["v_proj"].T).reshape(T, g.n_kv_heads, g.head_dim)
        q = rms_norm(q, w["q_norm"], g.rms_eps)
        k = rms_norm(k, w["k_norm"], g.rms_eps)
        q = rope_neox(q, positions, g.rope_theta)
        k = rope_neox(k, positions, g.rope_theta)
        return q, k, v

    def post_attention(self, l, x, attn):
        """o_proj + residual, post-norm, SwiGLU MLP + residual. attn: [T, nq*hd]."""
        g, w = self.g, self.layers[l]
        x = x + attn @ w["o_proj"].T
        h2 = rms_norm(x, w["post_norm"], g.rms_eps)
        a = silu(h2 @ w["gate_proj"].T) * (h2 @ w["up_proj"].T)
        return x + a @ w["down_proj"].T

    def head(self, x, head_w=None):
        """Final RMSNorm and codec_head (talker_forward_core). Returns (hidden, logits).

        head_w [V, H] replaces codec_head: the code predictor of the rightkit-qts page
        ("tts_transformer.rs", forward_code_pred_prefill_cached / forward_code_pred_step_cached)
        projects its prefill with heads[0] and generation step g with heads[g]."""
        y = rms_norm(x, self.final_norm, self.g.rms_eps)
        W = self.codec_head if head_w is None else np.asarray(head_w, F64)
        return y, y @ W.T

    # -- mode A: uncached full-sequence forward ---------------------------------
    def forward_full(self, emb, return_layers=False):
        """Every row of emb[T, H] at positions 0..T-1 with an explicit T x T causal mask.

        Returns (hidden [T,H], logits [T,V]) and, with return_layers, the residual
        stream after each layer [n_layers, T, H].
        """
        g = self.g
        x = np.asarray(emb, F64)
        T = x.shape[0]
        pos = np.arange(T)
        mask = np.where(pos[None, :] <= pos[:, None], 0.0, -np.inf)      # [q, k]
        group = g.n_q_heads // g.n_kv_heads
        taps = []
        for l in range(g.n_layers):
            q, k, v = self.qkv(l, x, pos)
            attn = np.empty((T, g.n_q_heads, g.head_dim), F64)
            for h in range(g.n_q_heads):
                kv = h // group
                s = (q[:, h, :] @ k[:, kv, :].T) / np.sqrt(F64(g.head_dim)) + mask
                attn[:, h, :] = softmax(s, axis=-1) @ v[:, kv, :]
            x = self.post_attention(l, x, attn.reshape(T, -1))
            if return_layers:
                taps.append(x.copy())
        hid, logits = self.head(x)
        if return_layers:
            return hid, logits, np.stack(taps)
        return hid, logits


# ----------------------------------------------------------------------------- Q8_0 KV storage

Q8_BLOCK = 32


def q8_0_quantize(x):
    """ggml Q8_0 (the cache storage type the qwen3-tts talker casts from): blocks of 32 along the
    last axis; d = max|x| / 127 in f32, codes = round-half-away-from-zero(x * (1/d)) in f32 (0 for
    an all-zero block), d stored as fp16 (nearest even). Returns (codes int8 [..., n], d fp16
    [..., n / 32])."""
    x32 = np.asarray(x, np.float32)
    shp = x32.shape
    if shp[-1] % Q8_BLOCK:
        raise ValueError("last axis must be a multiple of 32")
    b = x32.reshape(shp[:-1] + (shp[-1] // Q8_BLOCK, Q8_BLOCK))
    amax = np.max(np.abs(b), axis=-1, keepdims=True)
    d = amax / np.float32(127.0)
    safe = np.where(d > 0, d, np.float32(1.0))
    inv = np.where(d > 0, np.float32(1.0) / safe, np.float32(0.0)).astype(np.float32)
    t = (b * inv).astype(np.float32)
    # half away from zero; the fractional part of an f32 below 2^23 is exact, so no add-then-floor
    # rounding error can move a value across the .5 boundary
    a = np.abs(t)
    fl = np.floor(a)
    q = np.sign(t) * np.where(a - fl >= np.float32(0.5), fl + 1, fl)
    return q.astype(np.int8).reshape(shp), d[..., 0].astype(np.float16)


def q8_0_dequantize(codes, d):
    """codes int8 [..., n], d fp16 [..., n / 32] -> fp64 values codes * d."""
    c = np.asarray(codes, F64)
    shp = c.shape
    b = c.reshape(shp[:-1] + (shp[-1] // Q8_BLOCK, Q8_BLOCK))
    return (b * np.asarray(d, np.float16).astype(F64)[..., None]).reshape(shp)


def q8_0_roundtrip(x):
    return q8_0_dequantize(*q8_0_quantize(x))


class OracleCache:
    """Mode B: the incremental KV-cached forward over n_streams independent streams.

    Cache layout per stream: K, V fp64 [n_layers, n_kv, max_seq_len, hd]; cur_len[s]
    counts the valid rows. Errors raise ValueError and leave the state unchanged.
    """

    def __init__(self, oracle: Oracle, n_streams: int, max_seq_len: int, round_kv=None, kv_q8=False):
        g = oracle.g
        self.o = oracle
        self.max_seq_len = max_seq_len
        shape = (g.n_layers, g.n_kv_heads, max_seq_len, g.head_dim)
        self.K = [np.zeros(shape, F64) for _ in range(n_streams)]
        self.V = [np.zeros(shape, F64) for _ in range(n_streams)]
        self.cur_len = [0] * n_streams
        # Diagnosis only: a callable applied to K/V rows before they are stored.
        self.round_kv = round_kv
        # Q8_0 storage (qwen3-tts talker, TurboQuantQ8_0): rows are stored as Q8_0; a call
        # attends the rows cached by earlier calls dequantized and its own rows exactly.
        self.kv_q8 = kv_q8

    def _store(self, s, l, rows, k, v):
        if self.round_kv is not None:
            k, v = self.round_kv(k), self.round_kv(v)
        if self.kv_q8:
            k, v = q8_0_roundtrip(k), q8_0_roundtrip(v)
        self.K[s][l][:, rows, :] = np.transpose(k, (1, 0, 2))
        self.V[s][l][:, rows, :] = np.transpose(v, (1, 0, 2))

    def rewind(self, s, new_len):
        if not 0 <= new_len <= self.cur_len[s]:
            raise ValueError("rewind length out of range")
        self.cur_len[s] = new_len

    def kv_import(self, s, k, v, length):
        """k, v: [n_layers, n_kv, length, hd]; sets cur_len[s] = length."""
        if length > self.max_seq_len:
            raise ValueError("import exceeds max_seq_len")
        k, v = np.asarray(k, F64), np.asarray(v, F64)
        if self.kv_q8:
            k, v = q8_0_roundtrip(k), q8_0_roundtrip(v)
        self.K[s][:, :, :length] = k
        self.V[s][:, :, :length] = v
        self.cur_len[s] = length

    def kv_export(self, s, length):
        return self.K[s][:, :, :length].copy(), self.V[s][:, :, :length].copy()

    def append_rows(self, s, emb, head_w=None):
        """talker_forward_core with n_past = cur_len[s]: T rows appended, all rows' outputs.
        head_w: another output head (see Oracle.head), else codec_head."""
        o, g = self.o, self.o.g
        x = np.asarray(emb, F64)
        T = x.shape[0]
        n_past = self.cur_len[s]
        if n_past + T > self.max_seq_len:
            raise ValueError("cache overflow")
        pos = n_past + np.arange(T)
        group = g.n_q_heads // g.n_kv_heads
        for l in range(g.n_layers):
            q, k, v = o.qkv(l, x, pos)
            # the call's own rows enter exactly, earlier rows as stored
            Kc = np.concatenate([self.K[s][l][:, :n_past], np.transpose(k, (1, 0, 2))], axis=1)
            Vc = np.concatenate([self.V[s][l][:, :n_past], np.transpose(v, (1, 0, 2))], axis=1)
            self._store(s, l, pos, k, v)
            attn = np.empty((T, g.n_q_heads, g.head_dim), F64)
            for h in range(g.n_q_heads):
                kv = h // group
                keys = Kc[kv, :n_past + T]                                   # [n_past+T, hd]
                sc = (q[:, h, :] @ keys.T) / np.sqrt(F64(g.head_dim))       # [T, n_past+T]
                vis = np.arange(n_past + T)[None, :] <= pos[:, None]
                sc = np.where(vis, sc, -np.inf)
                attn[:, h, :] = softmax(sc, axis=-1) @ Vc[kv, :n_past + T]
            x = o.post_attention(l, x, attn.reshape(T, -1))
        hid, logits = o.head(x, head_w)
        self.cur_len[s] = n_past + T
        return hid, logits

    def prefill(self, s, emb, head_w=None):
        """talker_forward_prefill: rewind to 0, append T rows, return the last row (hidden, logits)."""
        T = np.asarray(emb).shape[0]
        if T < 1 or T > self.max_seq_len:
            raise ValueError("prefill length out of range")
        self.cur_len[s] = 0
        hid, logits = self.append_rows(s, emb, head_w)
        return hid[-1], logits[-1]

    def decode(self, embs, head_w=None):
        """talker_forward_decode over streams 0..B-1, one row each. Returns (hidden [B,H], logits [B,V]).
        head_w: another output head (see Oracle.head), else codec_head."""
        o, g = self.o, self.o.g
        x = np.asarray(embs, F64)
        B = x.shape[0]
        for s in range(B):
            if self.cur_len[s] + 1 > self.max_seq_len:
                raise ValueError("decode would overflow the cache")
        pos = np.array([self.cur_len[s] for s in range(B)])
        for l in range(g.n_layers):
            q, k, v = o.qkv(l, x, pos)
            attn = np.empty((B, g.n_q_heads, g.head_dim), F64)
            for s in range(B):
                Ks = np.concatenate([self.K[s][l][:, :pos[s]], np.transpose(k[s:s + 1], (1, 0, 2))], axis=1)
                Vs = np.concatenate([self.V[s][l][:, :pos[s]], np.transpose(v[s:s + 1], (1, 0, 2))], axis=1)
                self._store(s, l, pos[s:s + 1], k[s:s + 1], v[s:s + 1])
                attn[s] = attend_one(q[s], Ks, Vs, pos[s] + 1)
            x = o.post_attention(l, x, attn.reshape(B, -1))
        hid, logits = o.head(x, head_w)
        for s in range(B):
            self.cur_len[s] += 1
        return hid, logits


def decode_row_lazy_cache(oracle: Oracle, x, pos, kv_layer):
    """One decode row at position pos against a cache whose rows [0, pos) come from kv_layer(l).

    kv_layer(l) returns (K, V) of layer l as [n_kv, >= pos, hd] arrays (the stored cache
    values); the row's own k, v are appended at pos as in talker_forward_decode. Layers are
    generated one at a time, so a long cache never has to be held for all layers at once.
    Returns (hidden [H], logits [V]).
    """
    g = oracle.g
    x = np.asarray(x, F64).reshape(1, -1)
    for l in range(g.n_layers):
        q, k, v = oracle.qkv(l, x, np.array([pos]))
        Kp, Vp = kv_layer(l)
        K = np.concatenate([np.asarray(Kp[:, :pos], F64), np.transpose(k, (1, 0, 2))], axis=1)
        V = np.concatenate([np.asarray(Vp[:, :pos], F64), np.transpose(v, (1, 0, 2))], axis=1)
        attn = attend_one(q[0], K, V, pos + 1)
        x = oracle.post_attention(l, x, attn.reshape(1, -1))
    hid, logits = oracle.head(x)
    return hid[0], logits[0]


# ----------------------------------------------------------------------------- TTS loop input / output

def embed_codes(tables, ids, overlay=None):
    """Decode input rows from codebook ids (talker_forward_core batch input, "input_embed").

    tables: list of G arrays [V_g, H] (table 0 = codec_embedding, then the acoustic tables);
    ids: int array [G, N], group-major (ids[g, n] is slot n's code in codebook g);
    overlay: [N, H] or None. Row n = sum_g tables[g][ids[g, n]] + overlay[n], in fp64.
    """
    ids = np.asarray(ids)
    G, N = ids.shape
    H = np.asarray(tables[0]).shape[1]
    x = np.zeros((N, H), F64)
    for g in range(G):
        x += np.asarray(tables[g], F64)[ids[g]]
    if overlay is not None:
        x += np.asarray(overlay, F64)
    return x


def code_predictor_frame(cache, emb, tables, table_of_step, heads, codes=None):
    """One frame of the code predictor on stream 0 of `cache` (rightkit-qts "tts_transformer.rs",
    predict_remaining_codebooks_kv_with_cache): prefill with emb [T0, H] and take the greedy code
    of its last row through heads[0]; then step i (generation step i + 1) reads row code_i of
    tables[table_of_step[i]], is decoded, and its code i + 1 is the greedy token of heads[i + 1].
    heads: len(table_of_step) + 1 arrays [V, H]. codes: optional codes to feed instead of the
    oracle's own (teacher forcing: codes[i] is the input of step i).
    Returns (logits [n_steps + 1, V], the oracle's greedy codes [n_steps + 1])."""
    _, lg = cache.prefill(0, emb, heads[0])
    logits, own = [lg], [argmax_low(lg)]
    for i, tab in enumerate(table_of_step):
        prev = own[i] if codes is None else int(codes[i])
        x = np.asarray(tables[tab], F64)[prev][None]
        _, lg = cache.decode(x, heads[i + 1])
        logits.append(lg[0])
        own.append(argmax_low(lg[0]))
    return np.stack(logits), np.array(own)


def suppress_logits(logits, vocab_tail, eos_id):
    """Codebook-0 logit suppression before selection: every token index >= V - vocab_tail except
    eos_id gets -inf (qwen3-tts talker prefill/step, "suppress_start"). Returns a copy."""
    out = np.array(logits, F64, copy=True)
    V = out.shape[-1]
    start = max(0, V - vocab_tail)
    keep = out[..., eos_id].copy() if 0 <= eos_id < V else None
    out[..., start:] = -np.inf
    if keep is not None and eos_id >= start:
        out[..., eos_id] = keep
    return out
