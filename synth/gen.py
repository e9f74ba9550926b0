"""Seeded generators and block encoders for the MoE layer workloads.

Weights are drawn N(0, std) in float32 and encoded into canonical blocks:

* GGUF Q4_0 block (18 bytes): little-endian fp16 scale ``d`` then 16 bytes of
  codes; element ``i < 16`` is the low nibble of code byte ``i`` and element
  ``i >= 16`` the high nibble of code byte ``i - 16``.  A decoder maps a code
  ``q`` to ``(q - 8) * d``.  (GGUF is the llama.cpp format the FreeToken pages
  name: "FreeToken：在桌面运行大规模模型的本地推理引擎", section 开源生态中的位置,
  and the Q4_0 bank of "深入FreeToken架构…全链路剖析" §五/§六.)
* OCP MXFP4 block (17 bytes): one E8M0 scale byte then 16 code bytes in the
  same nibble order; codes are E2M1 (OCP Microscaling Formats v1.0).

The encoders below only produce bytes; decoding them is the job of the oracle
on one side and the CUDA kernels on the other.
"""
from __future__ import annotations

import dataclasses
import math
import zlib
from concurrent.futures import ThreadPoolExecutor

import numpy as np

QTYPE_BLOCK_BYTES = {"q4_0": 18, "mxfp4": 17, "nvfp4": 9, "mxfp8": 33}
QTYPE_BLOCK_ELEMS = {"q4_0": 32, "mxfp4": 32, "nvfp4": 16, "mxfp8": 32}
BLOCK = 32

# Workloads: the shapes, value distributions and seeds of the layer configs.
CONFIGS = {
    "tiny": dict(H=256, I=128, E=8, k=2, T=64, qtype="q4_0", zipf=0.0, no_ties=True, seed=0),
    "decode": dict(H=2048, I=768, E=128, k=8, T=64, T_sweep=(1, 4, 16, 64), qtype="q4_0",
                   qtypes=("q4_0", "mxfp4", "nvfp4", "mxfp8"),
                   zipf=0.0, no_ties=False, seed=0),
    "prefill": dict(H=2048, I=768, E=128, k=8, T=4096, qtype="q4_0", qtypes=("q4_0", "mxfp4", "nvfp4", "mxfp8"),
                    zipf=1.0, no_ties=False, seed=0),
    "large": dict(H=7168, I=2048, E=256, k=8, T=2048, T_total=16384, decode_T=32, qtype="mxfp4",
                  shared=True, zipf=1.0, no_ties=False, seed=0),
    "stream": dict(H=2048, I=768, E=128, k=8, T=1, layers=48, slots=32, steps=2048, p_repeat=0.7,
                   qtype="q4_0", zipf=1.0, seed=0),
}


def _rng(seed: int, *tags) -> np.random.Generator:
    """Independent stream per (seed, tags); tags may be strings or ints."""
    ent = [int(seed) & 0xFFFFFFFF]
    for t in tags:
        ent.append(zlib.crc32(t.encode()) if isinstance(t, str) else int(t) & 0xFFFFFFFF)
    return np.random.default_rng(ent)


# ----------------------------------------------------------------------------- bf16 inputs
def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (round to nearest even); returns the uint16 bit patterns."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def gen_x_bf16(seed: int, T: int, H: int, tag: str = "x") -> np.ndarray:
    """Activations ~N(0,1) rounded to bf16; uint16 bits [T, H]."""
    x = _rng(seed, tag, T, H).standard_normal((T, H), dtype=np.float32)
    return f32_to_bf16_bits(x)


def gen_gate_weights(seed: int, E: int, H: int, tag: str = "gate") -> np.ndarray:
    """Router gate matrix ~N(0, 1/H) rounded to bf16 (logits of unit scale for unit
    activations); uint16 bits [E, H]."""
    w = _rng(seed, tag, E, H).standard_normal((E, H), dtype=np.float32) / np.float32(np.sqrt(H))
    return f32_to_bf16_bits(w)


def zipf_bias(E: int, s: float) -> np.ndarray:
    """Expert popularity skew added to router logits: -s * ln(e + 1) (expert 0 most popular)."""
    return -s * np.log(np.arange(1, E + 1, dtype=np.float64))


def gen_logits(seed: int, T: int, E: int, zipf: float = 0.0, no_ties: bool = False,
               tag: str = "logits") -> np.ndarray:
    """Router logits fp32 [T, E] = N(0,1) (+ log-Zipf bias).  With ``no_ties`` a token's
    row is redrawn until its E values are pairwise distinct."""
    rng = _rng(seed, tag, T, E)
    lg = rng.standard_normal((T, E), dtype=np.float32)
    if no_ties:
        for t in range(T):
            while len(np.unique(lg[t])) != E:
                lg[t] = rng.standard_normal(E, dtype=np.float32)
    if zipf:
        lg = (lg.astype(np.float64) + zipf_bias(E, zipf)[None, :]).astype(np.float32)
    return lg


# ----------------------------------------------------------------------------- encoders
def quantize_q4_0(w: np.ndarray) -> np.ndarray:
    """Encode float32 [..., K] (K % 32 == 0) into Q4_0 blocks uint8 [..., K/32, 18].

    Per block: m = the element of largest magnitude (first on ties), d = m / -8,
    q = clamp(floor(x * (1/d) + 8.5), 0, 15); d is stored as fp16 (round to nearest).
    An all-zero block stores d = 0 and q = 8."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    K = w.shape[-1]
    assert K % BLOCK == 0
    lead = w.shape[:-1]
    b = w.reshape(-1, BLOCK)
    n = b.shape[0]
    idx = np.argmax(np.abs(b), axis=1)
    m = b[np.arange(n), idx]
    d = (m / np.float32(-8.0)).astype(np.float32)
    with np.errstate(divide="ignore"):
        inv = np.where(d != 0, np.float32(1.0) / np.where(d != 0, d, 1), np.float32(0)).astype(np.float32)
    q = np.clip(np.floor(b * inv[:, None] + np.float32(8.5)), 0, 15).astype(np.uint8)
    out = np.empty((n, 18), dtype=np.uint8)
    out[:, 0:2] = d.astype(np.float16).view(np.uint8).reshape(n, 2)
    out[:, 2:18] = q[:, :16] | (q[:, 16:] << 4)
    return out.reshape(*lead, K // BLOCK, 18)


_E2M1_GRID = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], dtype=np.float64)


def quantize_mxfp4(w: np.ndarray) -> np.ndarray:
    """Encode float32 [..., K] into MXFP4 blocks uint8 [..., K/32, 17].

    Per block: shared exponent u = floor(log2(amax)) - 2 clamped to [-127, 127]
    (scale byte u + 127; amax == 0 gives byte 127 and zero codes); each element
    x / 2^u is rounded to the nearest E2M1 magnitude (ties to the even code),
    saturating at 6; bit 3 of the code is the sign."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    K = w.shape[-1]
    assert K % BLOCK == 0
    lead = w.shape[:-1]
    flat = w.reshape(-1, BLOCK)
    if flat.shape[0] > (1 << 18):  # bound the temporaries: encode in slices of blocks
        parts = [quantize_mxfp4(flat[i:i + (1 << 18)]) for i in range(0, flat.shape[0], 1 << 18)]
        return np.concatenate(parts, axis=0).reshape(*lead, K // BLOCK, 17)
    b = flat.astype(np.float64)
    n = b.shape[0]
    amax = np.max(np.abs(b), axis=1)
    with np.errstate(divide="ignore"):
        u = np.where(amax > 0, np.floor(np.log2(np.where(amax > 0, amax, 1.0))) - 2, 0.0)
    u = np.clip(u, -127, 127)
    v = b / np.exp2(u)[:, None]
    mag = np.minimum(np.abs(v), 6.0)
    dist = np.abs(mag[..., None] - _E2M1_GRID)
    c = np.argmin(dist, axis=-1)  # lower code on a tie
    c1 = np.minimum(c + 1, 7)
    tie = (np.take_along_axis(dist, c1[..., None], -1)[..., 0] == np.take_along_axis(dist, c[..., None], -1)[..., 0]) & (c1 != c)
    c = np.where(tie & (c % 2 == 1), c1, c)  # round half to even code
    sign = ((v < 0) & (c != 0)).astype(np.uint8)
    code = (c.astype(np.uint8) | (sign << 3)).astype(np.uint8)
    out = np.empty((n, 17), dtype=np.uint8)
    out[:, 0] = (u + 127).astype(np.uint8)
    out[:, 1:17] = code[:, :16] | (code[:, 16:] << 4)
    return out.reshape(*lead, K // BLOCK, 17)


def _e4m3_grid() -> np.ndarray:
    """The 127 finite non-negative E4M3 values in code order (codes 0x00..0x7E)."""
    c = np.arange(127)
    e, m = c >> 3, c & 7
    return np.where(e == 0, m / 8.0 * 2.0 ** -6, np.exp2(e - 7.0) * (1.0 + m / 8.0))


_E4M3 = _e4m3_grid()


def _round_e4m3(x: np.ndarray) -> np.ndarray:
    """Codes (uint8, sign in bit 7) of the E4M3 values nearest to x, ties to the even
    code, saturating at 448."""
    x = np.asarray(x, dtype=np.float64)
    mag = np.minimum(np.abs(x), 448.0).reshape(-1)
    out = np.empty(mag.shape, dtype=np.uint8)
    for i in range(0, mag.size, 1 << 16):
        v = mag[i:i + (1 << 16)]
        hi = np.clip(np.searchsorted(_E4M3, v, side="left"), 0, 126)
        lo = np.clip(hi - 1, 0, 126)
        dlo, dhi = np.abs(v - _E4M3[lo]), np.abs(_E4M3[hi] - v)
        c = np.where(dhi < dlo, hi, lo)
        c = np.where((dhi == dlo) & (hi != lo), np.where(lo % 2 == 0, lo, hi), c)
        out[i:i + (1 << 16)] = c
    sign = ((x.reshape(-1) < 0) & (out != 0)).astype(np.uint8)
    return (out | (sign << 7)).reshape(x.shape)


def quantize_nvfp4(w: np.ndarray):
    """Encode float32 [..., K] (K % 16 == 0) into NVFP4: blocks uint8 [..., K/16, 9] and
    one fp32 tensor scale for the whole array.

    tensor_scale = amax / (6 * 448) (1 for an all-zero array); per 16-element block the
    scale byte is the E4M3 value nearest to block_amax / 6 / tensor_scale; each element
    x / (scale * tensor_scale) goes to the nearest E2M1 magnitude (ties to the even
    code), saturating at 6.  Element i < 8 is the low nibble of code byte i."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    K = w.shape[-1]
    assert K % 16 == 0
    lead = w.shape[:-1]
    b = w.reshape(-1, 16).astype(np.float64)
    n = b.shape[0]
    amax = float(np.max(np.abs(b))) if b.size else 0.0
    ts = np.float32(amax / (6.0 * 448.0)) if amax > 0 else np.float32(1.0)
    sbyte = _round_e4m3(np.max(np.abs(b), axis=1) / 6.0 / float(ts))
    sval = np.where(sbyte == 0, 0.0, _E4M3[sbyte & 0x7F])
    with np.errstate(divide="ignore", invalid="ignore"):
        v = np.where(sval[:, None] > 0, b / (sval[:, None] * float(ts)), 0.0)
    mag = np.minimum(np.abs(v), 6.0)
    dist = np.abs(mag[..., None] - _E2M1_GRID)
    c = np.argmin(dist, axis=-1)
    c1 = np.minimum(c + 1, 7)
    tie = (np.take_along_axis(dist, c1[..., None], -1)[..., 0] == np.take_along_axis(dist, c[..., None], -1)[..., 0]) & (c1 != c)
    c = np.where(tie & (c % 2 == 1), c1, c)
    sign = ((v < 0) & (c != 0)).astype(np.uint8)
    code = (c.astype(np.uint8) | (sign << 3)).astype(np.uint8)
    out = np.empty((n, 9), dtype=np.uint8)
    out[:, 0] = sbyte
    out[:, 1:9] = code[:, :8] | (code[:, 8:] << 4)
    return out.reshape(*lead, K // 16, 9), float(ts)


def quantize_mxfp8(w: np.ndarray) -> np.ndarray:
    """Encode float32 [..., K] into MXFP8 (E4M3) blocks uint8 [..., K/32, 33].

    Per block: shared exponent u = floor(log2(amax)) - 8 clamped to [-127, 127] (scale
    byte u + 127; amax == 0 gives byte 127 and zero elements); each element x / 2^u is
    rounded to the nearest E4M3 value (ties to the even code), saturating at 448."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    K = w.shape[-1]
    assert K % BLOCK == 0
    lead = w.shape[:-1]
    b = w.reshape(-1, BLOCK).astype(np.float64)
    n = b.shape[0]
    amax = np.max(np.abs(b), axis=1)
    with np.errstate(divide="ignore"):
        u = np.where(amax > 0, np.floor(np.log2(np.where(amax > 0, amax, 1.0))) - 8, 0.0)
    u = np.clip(u, -127, 127)
    out = np.empty((n, 33), dtype=np.uint8)
    out[:, 0] = (u + 127).astype(np.uint8)
    out[:, 1:] = _round_e4m3(b / np.exp2(u)[:, None])
    return out.reshape(*lead, K // BLOCK, 33)


_ENCODERS = {"q4_0": quantize_q4_0, "mxfp4": quantize_mxfp4, "nvfp4": quantize_nvfp4,
             "mxfp8": quantize_mxfp8}


def gen_expert_weights(seed: int, tag: str, E: int, N: int, K: int, qtype: str,
                       std: float = 0.02, distinct: int | None = None,
                       threads: int = 8) -> np.ndarray:
    """Canonical block bytes uint8 [E, N, K/block, block bytes] (see
    gen_expert_weights_ts, which also returns NVFP4's per-matrix tensor scales)."""
    return gen_expert_weights_ts(seed, tag, E, N, K, qtype, std, distinct, threads)[0]


def gen_expert_weights_ts(seed: int, tag: str, E: int, N: int, K: int, qtype: str,
                          std: float = 0.02, distinct: int | None = None, threads: int = 8):
    """Canonical block bytes uint8 [E, N, K/block, block bytes] of N(0, std) weights, and
    for NVFP4 the fp32 tensor scale of every expert's matrix (float32 [E]; None for the
    formats without one).

    Expert e draws from its own stream (seed, tag, e).  With ``distinct`` < E only that
    many expert matrices are drawn (used for the largest banks, where drawing every
    expert would dominate run time); expert e then holds draw src[e] with its rows in a
    seeded order of its own, where src is a seeded permutation of the experts taken
    modulo ``distinct``.  Rows of a draw are independent N(0, std) rows, so every expert
    keeps the distribution, and no two experts hold the same matrix."""
    enc = _ENCODERS[qtype]
    nb = QTYPE_BLOCK_BYTES[qtype]
    out = np.empty((E, N, K // QTYPE_BLOCK_ELEMS[qtype], nb), dtype=np.uint8)
    ts = np.ones(E, dtype=np.float32) if qtype == "nvfp4" else None
    D = E if distinct is None else min(distinct, E)

    def one(e):
        w = _rng(seed, tag, qtype, e, N, K).standard_normal((N, K), dtype=np.float32)
        w *= np.float32(std)
        if qtype == "nvfp4":
            out[e], ts[e] = enc(w)
        else:
            out[e] = enc(w)

    with ThreadPoolExecutor(max_workers=threads) as ex:
        list(ex.map(one, range(D)))
    if D < E:
        draws = out[:D].copy()
        src = _rng(seed, tag, "expert_src", E, D).permutation(E) % D

        draws_ts = ts[:D].copy() if ts is not None else None

        def place(e):
            rows = _rng(seed, tag, "expert_rows", e, N).permutation(N)
            out[e] = draws[src[e]][rows]
            if ts is not None:
                ts[e] = draws_ts[src[e]]

        with ThreadPoolExecutor(max_workers=threads) as ex:
            list(ex.map(place, range(E)))
    return out, ts


@dataclasses.dataclass
class LayerInputs:
    """One layer's inputs in canonical form (host numpy)."""
    H: int
    I: int
    E: int
    k: int
    T: int
    qtype: str
    x: np.ndarray          # uint16 bf16 bits [T, H]
    logits: np.ndarray     # float32 [T, E]
    w13: np.ndarray        # uint8 [E, 2I, H/32, blk]; rows [0, I) gate, [I, 2I) up
    w2: np.ndarray         # uint8 [E, H, I/32, blk]
    shared_w13: np.ndarray | None = None  # uint8 [1, 2I, H/32, blk]
    shared_w2: np.ndarray | None = None   # uint8 [1, H, I/32, blk]
    # NVFP4 only: fp32 tensor scale of each expert's matrix
    w13_ts: np.ndarray | None = None      # float32 [E]
    w2_ts: np.ndarray | None = None       # float32 [E]
    shared_w13_ts: np.ndarray | None = None
    shared_w2_ts: np.ndarray | None = None

    @property
    def ts(self):
        """The tensor scales as the oracle's layer takes them (None for formats without)."""
        if self.w13_ts is None:
            return None
        return {"w13": self.w13_ts, "w2": self.w2_ts, "shared_w13": self.shared_w13_ts,
                "shared_w2": self.shared_w2_ts}


def make_layer(H: int, I: int, E: int, k: int, T: int, qtype: str = "q4_0", seed: int = 0,
               zipf: float = 0.0, no_ties: bool = False, shared: bool = False,
               distinct: int | None = None, std: float = 0.02, x_tag: str = "x",
               logit_tag: str = "logits", **_unused) -> LayerInputs:
    w13, w13_ts = gen_expert_weights_ts(seed, "w13", E, 2 * I, H, qtype, std, distinct)
    w2, w2_ts = gen_expert_weights_ts(seed, "w2", E, H, I, qtype, std, distinct)
    sw13 = sw2 = sw13_ts = sw2_ts = None
    if shared:
        sw13, sw13_ts = gen_expert_weights_ts(seed, "shared_w13", 1, 2 * I, H, qtype, std)
        sw2, sw2_ts = gen_expert_weights_ts(seed, "shared_w2", 1, H, I, qtype, std)
    return LayerInputs(H, I, E, k, T, qtype,
                       gen_x_bf16(seed, T, H, x_tag),
                       gen_logits(seed, T, E, zipf, no_ties, logit_tag),
                       w13, w2, sw13, sw2, w13_ts, w2_ts, sw13_ts, sw2_ts)


def stream_trace(seed: int, steps: int, layers: int, E: int, k: int, p_repeat: float,
                 s: float) -> np.ndarray:
    """Batch-1 decode expert trace int32 [steps, layers, k].

    Step 0 draws; afterwards each (step, layer) repeats that layer's previous ids with
    probability p_repeat, else draws k distinct ids from Zipf(s) over E experts by
    rejection (redraw an id already taken)."""
    rng = _rng(seed, "trace", steps, layers, E, k)
    p = 1.0 / np.power(np.arange(1, E + 1, dtype=np.float64), s)
    cdf = np.cumsum(p / p.sum())
    out = np.empty((steps, layers, k), dtype=np.int32)
    for st in range(steps):
        for l in range(layers):
            if st > 0 and rng.random() < p_repeat:
                out[st, l] = out[st - 1, l]
                continue
            got: list[int] = []
            while len(got) < k:
                e = int(np.searchsorted(cdf, rng.random(), side="right"))
                e = min(e, E - 1)
                if e not in got:
                    got.append(e)
            out[st, l] = got
    return out
