"""Seeded synthetic inputs for the lookahead sparse decode step.

This module is the one place that both the CUDA path and the CPU oracle take
their inputs from.  It holds no arithmetic of the method itself (no scoring,
selection, table update or attention); it only draws keys, values, queries,
planted "hot" blocks and initial resident sets from a seed.

Determinism across devices
--------------------------
Bulk keys and values are drawn with a counter-based generator that is
bit-identical in numpy (host) and torch (device):

* ``mix32`` is a 32-bit integer bijection (xor-shift / multiply rounds with
  odd constants below 2**31, so every product fits a signed 64-bit integer and
  torch's int64 arithmetic never overflows);
* a chunk key absorbs (seed, stream, layer, request, head) through ``mix32``;
* element ``i`` of a chunk draws ``mix32(mix32(i ^ key) ^ key2) >> 16`` and
  looks it up in a 65536-entry inverse-normal table (``NORMAL_TABLE``), i.e. an
  N(0,1) sample quantised to 2**-16 in probability;
* planted shifts are added in float32 (one IEEE add, identical on both sides)
  and the result is rounded to bfloat16 with round-to-nearest-even.

Small per-head quantities (unit directions, queries, hot-block sets, initial
resident sets) are computed on the host in float64/float32 and uploaded.

Workload recipe (shapes of the Qwen3-8B / Qwen3-32B / Llama-3.1-8B decode
experiments named on the OasisKV pages, Fig. 2, Table 1 and Table 2 captions):
K, V ~ N(0,1); per (layer, request, KV head) a unit vector u; every key of a
hot block gets +3u; the true query of each query head in the GQA group is
2u + e with e ~ N(0,1) drifting across decode steps as AR(1) with coefficient
rho; lookahead query j is the true query plus N(0, 0.3**2) noise.

Drifting hot set (``hot_mode="drift"``, the long-output reasoning workload of
Table 1's long-output rows): per (layer, request, KV head) a plane spanned by
two orthonormal vectors a, c and a pool of ``n_pool`` planted blocks; pool
block i (in draw order) has its own direction v_i = cos(phi_i) a + sin(phi_i) c,
phi_i = 2 pi i / n_pool, and each of its keys gets +3 v_i.  The query
direction u_s drifts as an AR(1) process on that great circle: a 2-vector
w_s = rho_u w_{s-1} + sqrt(1 - rho_u**2) xi_s (w_0, xi_s ~ N(0, I_2)),
u_s = (w_s / |w_s|) . [a; c].  The true query is 2 u_s + e_s as above.  The hot
set at step s is the ``n_hot`` pool blocks best aligned with u_s; rho_u = 0.997
makes it turn over by about 5% per step (see :func:`hot_set_turnover`).
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional, Sequence

import numpy as np

M32 = 0xFFFFFFFF
_C1 = 0x21F0AAAD
_C2 = 0x735A2D97
_K2_SALT = 0x5BD1E995

STREAM_K = 0
STREAM_V = 1
STREAM_U = 2
STREAM_QNOISE = 3
STREAM_LANOISE = 4
STREAM_APPEND_K = 5
STREAM_APPEND_V = 6
STREAM_PLANE_C = 7      # second vector of the drift plane
STREAM_UDRIFT = 8       # the 2-D AR(1) draws of the drifting query direction


# --------------------------------------------------------------------------
# counter-based generator (numpy side)
# --------------------------------------------------------------------------
def mix32_np(x: np.ndarray) -> np.ndarray:
    """32-bit integer bijection, elementwise; returns uint32 (the input is taken
    mod 2**32).  uint32 products wrap mod 2**32, as the definition wants."""
    x = np.asarray(x)
    x = (x & np.uint64(M32)).astype(np.uint32) if x.dtype != np.uint32 else x.copy()
    x ^= x >> np.uint32(16)
    x *= np.uint32(_C1)
    x ^= x >> np.uint32(15)
    x *= np.uint32(_C2)
    x ^= x >> np.uint32(15)
    return x


def mix32_int(x: int) -> int:
    x &= M32
    x ^= x >> 16
    x = (x * _C1) & M32
    x ^= x >> 15
    x = (x * _C2) & M32
    x ^= x >> 15
    return x


def chunk_key(seed: int, stream: int, layer: int, b: int, h: int) -> tuple:
    k = mix32_int(seed & M32)
    for v in (stream, layer, b, h):
        k = mix32_int(k ^ (v & M32))
    return k, mix32_int(k ^ _K2_SALT)


def _normal_table() -> np.ndarray:
    from scipy.special import ndtri

    p = (np.arange(65536, dtype=np.float64) + 0.5) / 65536.0
    return ndtri(p).astype(np.float32)


NORMAL_TABLE = _normal_table()


def hash_normals(seed: int, stream: int, layer: int, b: int, h: int,
                 start: int, count: int) -> np.ndarray:
    """float32 N(0,1) draws for elements [start, start+count) of one chunk."""
    k1, k2 = chunk_key(seed, stream, layer, b, h)
    idx = (np.arange(start, start + count, dtype=np.uint64) & np.uint64(M32)).astype(np.uint32)
    v = mix32_np(mix32_np(idx ^ np.uint32(k1)) ^ np.uint32(k2))
    return NORMAL_TABLE[v >> np.uint32(16)]


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (round to nearest, ties to even); finite input."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    # uint32 wrap-around only drops bits above 2**32, which the shift and the
    # 16-bit result drop anyway
    r = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


# --------------------------------------------------------------------------
# workloads
# --------------------------------------------------------------------------
@dataclasses.dataclass
class Workload:
    name: str
    L: int
    B: int
    Hq: int
    Hkv: int
    ctx: List[int]            # per-request context length (tokens)
    Kb: int                   # token budget / block size
    C: int                    # fetch cap, blocks per KV head per step
    n_la: int = 4
    d: int = 128
    bs: int = 16
    n_hot: int = 16
    hot_mode: str = "random"  # "random" | "spans_sink_recent" | "drift"
    steps: int = 1
    rho: float = 0.9
    la_sigma: float = 0.3
    seed: int = 0
    nb_max: Optional[int] = None
    P: Optional[int] = None   # HBM slots per (layer, request, KV head)
    n_pool: int = 256         # planted blocks per head with their own direction ("drift")
    rho_u: float = 0.997      # AR(1) coefficient of the drifting query direction ("drift")

    def __post_init__(self):
        if len(self.ctx) != self.B:
            raise ValueError("ctx must list one context length per request")
        if self.hot_mode not in ("random", "spans_sink_recent", "drift"):
            raise ValueError(f"unknown hot_mode {self.hot_mode!r}")
        # planted blocks are drawn from the blocks of the starting context, so that
        # appends (which advance ctx in place) do not change them
        self.ctx0 = list(self.ctx)
        if self.nb_max is None:
            self.nb_max = max(-(-c // self.bs) for c in self.ctx)
        if self.P is None:
            self.P = self.Kb

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def T_max(self) -> int:
        return self.nb_max * self.bs

    def nb(self, b: int) -> int:
        return -(-self.ctx[b] // self.bs)

    def nb0(self, b: int) -> int:
        """Blocks of request b's starting context (the planted blocks lie among them)."""
        return -(-self.ctx0[b] // self.bs)


def fetch_cap_from_ratio(ratio: Optional[float], Kb: int) -> int:
    """Fetch ratio -> per-step cap in blocks: max(1, floor(ratio*Kb)); None = fetch all."""
    if ratio is None:
        return Kb
    return max(1, int(math.floor(ratio * Kb + 1e-9)))


def tiny(seed: int = 0) -> Workload:
    """1 layer, batch 1, 32/8 heads, d 128, ctx 4096, budget 512, cap 4, 16 hot blocks."""
    return Workload("tiny", L=1, B=1, Hq=32, Hkv=8, ctx=[4096], Kb=32, C=4,
                    n_hot=16, seed=seed, rho=0.9)


def qwen3_8b_decode(seed: int = 0, B: int = 32, L: int = 36, ctx: int = 32768) -> Workload:
    """Qwen3-8B decode shape: 36 layers, 32/8 heads, batch 32, ctx 32K, budget 2048, ratio 0.02."""
    return Workload("qwen3_8b_decode", L=L, B=B, Hq=32, Hkv=8, ctx=[ctx] * B, Kb=128,
                    C=fetch_cap_from_ratio(0.02, 128), n_hot=64, steps=64, seed=seed)


def llama31_8b_long(seed: int = 0, B: int = 8, L: int = 32, ctx: int = 131072) -> Workload:
    """Llama-3.1-8B long-input shape: 32 layers, batch 8, ctx 128K, ratio 0.05, span+sink hot set."""
    return Workload("llama31_8b_long", L=L, B=B, Hq=32, Hkv=8, ctx=[ctx] * B, Kb=128,
                    C=fetch_cap_from_ratio(0.05, 128), n_hot=64, hot_mode="spans_sink_recent",
                    steps=32, seed=seed)


def qwen3_32b(seed: int = 0, ratio: Optional[float] = 0.01, B: int = 16, L: int = 64,
              ctx: int = 32768) -> Workload:
    """Qwen3-32B shape: 64 layers, 64/8 heads (GQA 8), batch 16, ctx 32K, budget 2048."""
    return Workload("qwen3_32b", L=L, B=B, Hq=64, Hkv=8, ctx=[ctx] * B, Kb=128,
                    C=fetch_cap_from_ratio(ratio, 128), n_hot=64, steps=32, seed=seed)


def long_output_ctx(B: int, start: int = 8192, end: int = 32768, steps: int = 256) -> List[int]:
    """Staggered starting contexts of the long-output workload (one token appended per step)."""
    span = end - start - steps
    return [start + (r * span) // max(1, B - 1) for r in range(B)]


def long_output(seed: int = 0, B: int = 128, L: int = 36, steps: int = 256, rho_u: float = 0.997) -> Workload:
    """Long-output reasoning decode: Qwen3-8B shape, batch 128, ctx 8K..32K, ratio 0.02,
    a hot set of 64 blocks drifting through a pool of 256 planted blocks per head
    (about 5% of the hot set replaced per step at rho_u = 0.997)."""
    ctx = long_output_ctx(B, steps=steps)
    w = Workload("long_output", L=L, B=B, Hq=32, Hkv=8, ctx=ctx, Kb=128,
                 C=fetch_cap_from_ratio(0.02, 128), n_hot=64, hot_mode="drift", n_pool=256,
                 rho_u=rho_u, steps=steps, seed=seed, nb_max=-(-(max(ctx) + steps) // 16))
    return w


# --------------------------------------------------------------------------
# per-head draws (host)
# --------------------------------------------------------------------------
def pool_blocks(w: Workload, layer: int, b: int, h: int) -> np.ndarray:
    """The planted pool of a drifting-hot-set workload, in draw order (pool index i
    has direction angle 2 pi i / n_pool)."""
    nb = w.nb0(b)
    rng = np.random.default_rng([w.seed, 101, layer, b, h])
    return rng.choice(nb, size=min(w.n_pool, nb), replace=False).astype(np.int64)


def hot_blocks(w: Workload, layer: int, b: int, h: int) -> np.ndarray:
    """Sorted indices of the planted blocks of one (layer, request, KV head)
    (for ``hot_mode="drift"``: the whole pool)."""
    nb = w.nb0(b)
    rng = np.random.default_rng([w.seed, 101, layer, b, h])
    if w.hot_mode == "drift":
        return np.sort(pool_blocks(w, layer, b, h))
    if w.hot_mode == "random":
        n = min(w.n_hot, nb)
        return np.sort(rng.choice(nb, size=n, replace=False)).astype(np.int64)
    if w.hot_mode == "spans_sink_recent":
        ends = set(range(min(4, nb))) | set(range(max(0, nb - 4), nb))
        span_len = max(1, (w.n_hot - len(ends)) // 4)
        lo, hi = 4, nb - 4 - span_len
        chosen: List[int] = []
        tries = 0
        while len(chosen) < 4 and hi > lo and tries < 10000:
            tries += 1
            s = int(rng.integers(lo, hi + 1))
            if all(abs(s - c) >= span_len for c in chosen):
                chosen.append(s)
        blocks = set(ends)
        for s in chosen:
            blocks.update(range(s, s + span_len))
        return np.array(sorted(x for x in blocks if x < nb), dtype=np.int64)
    raise ValueError(w.hot_mode)


def unit_dir(w: Workload, layer: int, b: int, h: int) -> np.ndarray:
    """float32 unit vector u of one (layer, request, KV head)."""
    z = hash_normals(w.seed, STREAM_U, layer, b, h, 0, w.d).astype(np.float64)
    return (z / np.linalg.norm(z)).astype(np.float32)


def drift_plane(w: Workload, layer: int, b: int, h: int):
    """Orthonormal float64 pair (a, c) spanning the plane of the drifting direction."""
    a = hash_normals(w.seed, STREAM_U, layer, b, h, 0, w.d).astype(np.float64)
    a = a / np.linalg.norm(a)
    c = hash_normals(w.seed, STREAM_PLANE_C, layer, b, h, 0, w.d).astype(np.float64)
    c = c - (c @ a) * a
    return a, c / np.linalg.norm(c)


def pool_dirs(w: Workload, layer: int, b: int, h: int) -> np.ndarray:
    """float64 [n][d] directions of the planted pool (pool index i at angle 2 pi i / n_pool)."""
    a, c = drift_plane(w, layer, b, h)
    n = len(pool_blocks(w, layer, b, h))
    phi = 2.0 * np.pi * np.arange(n) / w.n_pool
    return np.cos(phi)[:, None] * a[None, :] + np.sin(phi)[:, None] * c[None, :]


def planted_shifts(w: Workload, layer: int, b: int, h: int):
    """(blocks int64 [n], float32 [n][d] shift added to every key of that block)."""
    if w.hot_mode == "drift":
        blocks = pool_blocks(w, layer, b, h)
        return blocks, (3.0 * pool_dirs(w, layer, b, h)).astype(np.float32)
    blocks = hot_blocks(w, layer, b, h)
    shift = (np.float32(3.0) * unit_dir(w, layer, b, h)).astype(np.float32)
    return blocks, np.repeat(shift[None, :], len(blocks), axis=0)


def _drift_w(w: Workload, layer: int, b: int, h: int, step: int) -> np.ndarray:
    """The 2-vector w_step of the AR(1) process of one head (float64)."""
    x = hash_normals(w.seed, STREAM_UDRIFT, layer, b, h, 0, 2).astype(np.float64)
    a = math.sqrt(1.0 - w.rho_u * w.rho_u)
    for s in range(1, step + 1):
        xi = hash_normals(w.seed, STREAM_UDRIFT, layer, b, h, 2 * s, 2).astype(np.float64)
        x = w.rho_u * x + a * xi
    return x


def _dir_from_w(x: np.ndarray, a: np.ndarray, c: np.ndarray) -> np.ndarray:
    """u = (x / |x|) . [a; c] for one 2-vector or rows of 2-vectors (float64)."""
    x = np.asarray(x, dtype=np.float64)
    n = np.sqrt(x[..., 0] * x[..., 0] + x[..., 1] * x[..., 1])
    return (x[..., 0] / n)[..., None] * a + (x[..., 1] / n)[..., None] * c


def query_dir(w: Workload, layer: int, b: int, h: int, step: int) -> np.ndarray:
    """float64 mean direction of the true queries of one head at a decode step."""
    if w.hot_mode != "drift":
        return unit_dir(w, layer, b, h).astype(np.float64)
    a, c = drift_plane(w, layer, b, h)
    return _dir_from_w(_drift_w(w, layer, b, h, step), a, c)


def hot_set(w: Workload, layer: int, b: int, h: int, step: int) -> List[int]:
    """The n_hot planted blocks best aligned with the query direction at `step`
    (sorted; alignment ties to the lower pool index).  For the fixed modes: the
    planted blocks themselves."""
    if w.hot_mode != "drift":
        return hot_blocks(w, layer, b, h).tolist()
    al = pool_dirs(w, layer, b, h) @ query_dir(w, layer, b, h, step)
    order = np.argsort(-al, kind="stable")[: w.n_hot]
    return sorted(pool_blocks(w, layer, b, h)[order].tolist())


def hot_set_turnover(w: Workload, layer: int, steps: int, heads=None) -> float:
    """Mean fraction of the hot set replaced per decode step, over `heads`
    ((request, KV head) pairs; default all) and steps 1..steps-1."""
    pairs = heads if heads is not None else [(b, h) for b in range(w.B) for h in range(w.Hkv)]
    if w.hot_mode != "drift":
        return 0.0
    tot, n = 0.0, 0
    for (b, h) in pairs:
        pool, dirs = pool_blocks(w, layer, b, h), pool_dirs(w, layer, b, h)
        a, c = drift_plane(w, layer, b, h)
        x = hash_normals(w.seed, STREAM_UDRIFT, layer, b, h, 0, 2).astype(np.float64)
        f = math.sqrt(1.0 - w.rho_u * w.rho_u)
        prev = None
        for s in range(steps):
            if s:
                x = w.rho_u * x + f * hash_normals(w.seed, STREAM_UDRIFT, layer, b, h, 2 * s, 2).astype(np.float64)
            order = np.argsort(-(dirs @ _dir_from_w(x, a, c)), kind="stable")[: w.n_hot]
            cur = set(pool[order].tolist())
            if prev is not None:
                tot += len(cur - prev) / max(1, len(cur))
                n += 1
            prev = cur
    return tot / max(1, n)


def head_kv_f32(w: Workload, layer: int, b: int, h: int, ntok: Optional[int] = None):
    """float32 keys/values of one head before bf16 rounding, tokens [0, ntok)."""
    if ntok is None:
        ntok = w.ctx[b]
    K = hash_normals(w.seed, STREAM_K, layer, b, h, 0, ntok * w.d).reshape(ntok, w.d)
    V = hash_normals(w.seed, STREAM_V, layer, b, h, 0, ntok * w.d).reshape(ntok, w.d)
    tok, rows = _planted_rows(w, layer, b, h, ntok)
    if len(tok):
        K[tok] = K[tok] + rows
    return K, V


def _planted_rows(w: Workload, layer: int, b: int, h: int, ntok: int):
    """Token indices < ntok of the planted blocks and the float32 shift of each."""
    blocks, shifts = planted_shifts(w, layer, b, h)
    tok = (blocks[:, None] * w.bs + np.arange(w.bs)[None, :]).reshape(-1)
    rows = np.repeat(shifts, w.bs, axis=0)
    keep = tok < ntok
    return tok[keep], rows[keep]


def head_kv(w: Workload, layer: int, b: int, h: int):
    """bf16 bit patterns [T_max][d] of K and V for one head; tokens >= ctx are zero."""
    Kf, Vf = head_kv_f32(w, layer, b, h)
    K = np.zeros((w.T_max, w.d), np.uint16)
    V = np.zeros((w.T_max, w.d), np.uint16)
    K[: w.ctx[b]] = f32_to_bf16_bits(Kf)
    V[: w.ctx[b]] = f32_to_bf16_bits(Vf)
    return K, V


def layer_kv(w: Workload, layer: int):
    """K, V bf16 bits [B][Hkv][T_max][d] for one layer (host; small workloads only)."""
    K = np.zeros((w.B, w.Hkv, w.T_max, w.d), np.uint16)
    V = np.zeros_like(K)
    for b in range(w.B):
        for h in range(w.Hkv):
            K[b, h], V[b, h] = head_kv(w, layer, b, h)
    return K, V


def _query_noise(w: Workload, layer: int, b: int, hq: int, step: int) -> np.ndarray:
    """AR(1) noise e_s of one query head (float64), e_0 ~ N(0, I)."""
    e = hash_normals(w.seed, STREAM_QNOISE, layer, b, hq, 0, w.d).astype(np.float64)
    a = math.sqrt(1.0 - w.rho * w.rho)
    for s in range(1, step + 1):
        xi = hash_normals(w.seed, STREAM_QNOISE, layer, b, hq, s * w.d, w.d).astype(np.float64)
        e = w.rho * e + a * xi
    return e


def head_queries(w: Workload, layer: int, b: int, h: int, step: int = 0):
    """True queries [G][d] and lookahead queries [n_la][G][d] (bf16 bits) of one KV head."""
    G, d = w.G, w.d
    u = query_dir(w, layer, b, h, step)
    q = np.zeros((G, d), np.float32)
    qla = np.zeros((w.n_la, G, d), np.float32)
    for g in range(G):
        hq = h * G + g
        qf = (2.0 * u + _query_noise(w, layer, b, hq, step)).astype(np.float32)
        q[g] = qf
        for j in range(w.n_la):
            xi = hash_normals(w.seed, STREAM_LANOISE, layer, b, hq,
                              (step * w.n_la + j) * d, d).astype(np.float64)
            qla[j, g] = (qf.astype(np.float64) + w.la_sigma * xi).astype(np.float32)
    return f32_to_bf16_bits(q), f32_to_bf16_bits(qla)


def layer_queries(w: Workload, layer: int, step: int = 0):
    """q bits [B][Hq][d] and q_la bits [B][n_la][Hq][d] for one layer and decode step."""
    q = np.zeros((w.B, w.Hq, w.d), np.uint16)
    qla = np.zeros((w.B, w.n_la, w.Hq, w.d), np.uint16)
    G = w.G
    for b in range(w.B):
        for h in range(w.Hkv):
            qh, qlah = head_queries(w, layer, b, h, step)
            q[b, h * G:(h + 1) * G] = qh
            qla[b, :, h * G:(h + 1) * G] = qlah
    return q, qla


def initial_resident(w: Workload, layer: int, b: int, h: int) -> np.ndarray:
    """Blocks resident in slots 0.. at the start (min(P, nb) random distinct blocks)."""
    nb = w.nb(b)
    n = min(w.P, nb)
    rng = np.random.default_rng([w.seed, 202, layer, b, h])
    return rng.choice(nb, size=n, replace=False).astype(np.int64)


def initial_tables(w: Workload, layer: int):
    """blk2slot [B][Hkv][nb_max], slot2blk [B][Hkv][P], last_used [B][Hkv][P] (int32)."""
    blk2slot = np.full((w.B, w.Hkv, w.nb_max), -1, np.int32)
    slot2blk = np.full((w.B, w.Hkv, w.P), -1, np.int32)
    last_used = np.full((w.B, w.Hkv, w.P), -1, np.int32)
    for b in range(w.B):
        for h in range(w.Hkv):
            res = initial_resident(w, layer, b, h)
            for p, x in enumerate(res):
                slot2blk[b, h, p] = x
                blk2slot[b, h, x] = p
    return blk2slot, slot2blk, last_used


def host_tier_from_kv(w: Workload, K: np.ndarray, V: np.ndarray) -> np.ndarray:
    """Pack K, V [B][Hkv][T_max][d] into the host tier layout [B][Hkv][nb_max][2][bs][d]."""
    B, H = K.shape[:2]
    k = K.reshape(B, H, w.nb_max, w.bs, w.d)
    v = V.reshape(B, H, w.nb_max, w.bs, w.d)
    return np.ascontiguousarray(np.stack([k, v], axis=3))


def pools_from_tables(w: Workload, host: np.ndarray, slot2blk: np.ndarray):
    """k_pool, v_pool [B][Hkv][P][bs][d] holding the resident blocks' K/V."""
    kp = np.zeros((w.B, w.Hkv, w.P, w.bs, w.d), np.uint16)
    vp = np.zeros_like(kp)
    for b in range(w.B):
        for h in range(w.Hkv):
            for p in range(w.P):
                x = slot2blk[b, h, p]
                if x >= 0:
                    kp[b, h, p] = host[b, h, x, 0]
                    vp[b, h, p] = host[b, h, x, 1]
    return kp, vp


# --------------------------------------------------------------------------
# counter-based generator (torch side): bit-identical to hash_normals
# --------------------------------------------------------------------------
def _mix32_torch(x):
    import torch  # noqa: F401

    x = x & M32
    x = x ^ (x >> 16)
    x = (x * _C1) & M32
    x = x ^ (x >> 15)
    x = (x * _C2) & M32
    x = x ^ (x >> 15)
    return x


_TABLE_CACHE = {}


def normal_table_torch(device):
    import torch

    key = str(device)
    if key not in _TABLE_CACHE:
        _TABLE_CACHE[key] = torch.from_numpy(NORMAL_TABLE.copy()).to(device)
    return _TABLE_CACHE[key]


def hash_normals_torch(seed: int, stream: int, layer: int, b: int, h: int,
                       start: int, count: int, device):
    """torch float32 version of :func:`hash_normals` (same bits on any device)."""
    import torch

    k1, k2 = chunk_key(seed, stream, layer, b, h)
    idx = torch.arange(start, start + count, dtype=torch.int64, device=device)
    v = _mix32_torch(_mix32_torch(idx ^ k1) ^ k2)
    return normal_table_torch(device)[v >> 16]


def head_kv_torch(w: Workload, layer: int, b: int, h: int, device):
    """bf16 K, V [T_max][d] of one head on ``device``; bit-identical to :func:`head_kv`."""
    import torch

    n = w.ctx[b] * w.d
    Kf = hash_normals_torch(w.seed, STREAM_K, layer, b, h, 0, n, device).view(w.ctx[b], w.d)
    Vf = hash_normals_torch(w.seed, STREAM_V, layer, b, h, 0, n, device).view(w.ctx[b], w.d)
    tok, rows = _planted_rows(w, layer, b, h, w.ctx[b])
    if len(tok):
        tok = torch.from_numpy(tok).to(device)
        Kf[tok] = Kf[tok] + torch.from_numpy(rows).to(device)
    K = torch.zeros((w.T_max, w.d), dtype=torch.bfloat16, device=device)
    V = torch.zeros_like(K)
    K[: w.ctx[b]] = Kf.to(torch.bfloat16)
    V[: w.ctx[b]] = Vf.to(torch.bfloat16)
    return K, V


# --------------------------------------------------------------------------
# vectorised draws (same bits as the per-head functions above)
# --------------------------------------------------------------------------
def _chunk_keys_multi(seed: int, stream: int, layer: int, bs_, hs_):
    k1 = np.array([chunk_key(seed, stream, layer, int(b), int(h))[0] for b, h in zip(bs_, hs_)], np.uint32)
    k2 = np.array([mix32_int(int(k) ^ _K2_SALT) for k in k1], np.uint32)
    return k1, k2


def hash_normals_multi(seed: int, stream: int, layer: int, bs_, hs_, start: int, count: int) -> np.ndarray:
    """[len(bs_)][count] float32 draws; row r equals hash_normals(..., bs_[r], hs_[r], start, count)."""
    k1, k2 = _chunk_keys_multi(seed, stream, layer, bs_, hs_)
    idx = (np.arange(start, start + count, dtype=np.uint64) & np.uint64(M32)).astype(np.uint32)[None, :]
    v = mix32_np(mix32_np(idx ^ k1[:, None]) ^ k2[:, None])
    return NORMAL_TABLE[v >> np.uint32(16)]


class _DriftDirs:
    """Per-step query directions of every head of one layer of a drifting-hot-set
    workload, [B*Hq][d] float64 (rows of one KV head repeated over its group);
    the same values as :func:`query_dir` step by step."""

    def __init__(self, w: Workload, layer: int):
        self.w, self.layer, self.step = w, layer, 0
        planes = [drift_plane(w, layer, b, h) for b in range(w.B) for h in range(w.Hkv)]
        self.a = np.stack([p[0] for p in planes])
        self.c = np.stack([p[1] for p in planes])
        self.bb = np.repeat(np.arange(w.B), w.Hkv)
        self.hh = np.tile(np.arange(w.Hkv), w.B)
        self.x = None

    def next(self) -> np.ndarray:
        w = self.w
        if self.x is None:
            self.x = hash_normals_multi(w.seed, STREAM_UDRIFT, self.layer, self.bb, self.hh, 0, 2).astype(np.float64)
        else:
            xi = hash_normals_multi(w.seed, STREAM_UDRIFT, self.layer, self.bb, self.hh,
                                    2 * self.step, 2).astype(np.float64)
            self.x = w.rho_u * self.x + math.sqrt(1.0 - w.rho_u * w.rho_u) * xi
        self.step += 1
        u = _dir_from_w(self.x, self.a, self.c)                      # [B*Hkv][d]
        return np.repeat(u, w.G, axis=0)


class QueryStream:
    """Queries of one layer for decode steps 0, 1, 2, ... (AR(1) noise carried over).

    ``next()`` returns (q bits [B][Hq][d], q_la bits [B][n_la][Hq][d]) and is
    bit-identical to :func:`layer_queries` for the same step.
    """

    def __init__(self, w: Workload, layer: int):
        self.w = w
        self.layer = layer
        self.step = 0
        B, Hq, d, G = w.B, w.Hq, w.d, w.G
        self.bb = np.repeat(np.arange(B), Hq)
        self.hq = np.tile(np.arange(Hq), B)
        self.drift = _DriftDirs(w, layer) if w.hot_mode == "drift" else None
        if self.drift is None:
            u = np.stack([unit_dir(w, layer, b, h) for b in range(B) for h in range(w.Hkv)])
            self.u = u.reshape(B, w.Hkv, 1, d).repeat(G, axis=2).reshape(B * Hq, d).astype(np.float64)
        self.e = None

    def next(self):
        w = self.w
        d = w.d
        if self.drift is not None:
            self.u = self.drift.next()
        if self.e is None:
            self.e = hash_normals_multi(w.seed, STREAM_QNOISE, self.layer, self.bb, self.hq, 0, d).astype(np.float64)
        else:
            a = math.sqrt(1.0 - w.rho * w.rho)
            xi = hash_normals_multi(w.seed, STREAM_QNOISE, self.layer, self.bb, self.hq,
                                    self.step * d, d).astype(np.float64)
            self.e = w.rho * self.e + a * xi
        qf = (2.0 * self.u + self.e).astype(np.float32)
        la = hash_normals_multi(w.seed, STREAM_LANOISE, self.layer, self.bb, self.hq,
                                self.step * w.n_la * d, w.n_la * d).astype(np.float64)
        la = la.reshape(-1, w.n_la, d)
        qla = (qf.astype(np.float64)[:, None, :] + w.la_sigma * la).astype(np.float32)
        self.step += 1
        q_bits = f32_to_bf16_bits(qf).reshape(w.B, w.Hq, d)
        qla_bits = f32_to_bf16_bits(qla).reshape(w.B, w.Hq, w.n_la, d).transpose(0, 2, 1, 3)
        return q_bits, np.ascontiguousarray(qla_bits)


def kv_request_torch(w: Workload, layer: int, b: int, device):
    """bf16 K, V [Hkv][T_max][d] of one request of one layer on ``device`` (same bits as head_kv)."""
    import torch

    H, n = w.Hkv, w.ctx[b] * w.d
    keys = [chunk_key(w.seed, STREAM_K, layer, b, h) for h in range(H)]
    vkeys = [chunk_key(w.seed, STREAM_V, layer, b, h) for h in range(H)]
    idx = torch.arange(0, n, dtype=torch.int64, device=device)[None, :]
    table = normal_table_torch(device)

    def draw(ks):
        k1 = torch.tensor([k[0] for k in ks], dtype=torch.int64, device=device)[:, None]
        k2 = torch.tensor([k[1] for k in ks], dtype=torch.int64, device=device)[:, None]
        v = _mix32_torch(_mix32_torch(idx ^ k1) ^ k2)
        return table[v >> 16].view(H, w.ctx[b], w.d)

    Kf = draw(keys)
    Vf = draw(vkeys)
    for h in range(H):
        tok, rows = _planted_rows(w, layer, b, h, w.ctx[b])
        if len(tok):
            tok = torch.from_numpy(tok).to(device)
            Kf[h, tok] = Kf[h, tok] + torch.from_numpy(rows).to(device)
    K = torch.zeros((H, w.T_max, w.d), dtype=torch.bfloat16, device=device)
    V = torch.zeros_like(K)
    K[:, : w.ctx[b]] = Kf.to(torch.bfloat16)
    V[:, : w.ctx[b]] = Vf.to(torch.bfloat16)
    return K, V


def append_tokens(w: Workload, layer: int, step: int):
    """Key/value rows (bf16 bits [B][Hkv][d]) appended at decode step `step`: N(0,1) draws."""
    k = np.stack([np.stack([hash_normals(w.seed, STREAM_APPEND_K, layer, b, h, step * w.d, w.d)
                            for h in range(w.Hkv)]) for b in range(w.B)])
    v = np.stack([np.stack([hash_normals(w.seed, STREAM_APPEND_V, layer, b, h, step * w.d, w.d)
                            for h in range(w.Hkv)]) for b in range(w.B)])
    return f32_to_bf16_bits(k), f32_to_bf16_bits(v)


def hash_normals_multi_torch(seed: int, stream: int, layer: int, bs_, hs_, start: int, count: int, device):
    """torch version of :func:`hash_normals_multi` (same bits on any device)."""
    import torch

    k1, k2 = _chunk_keys_multi(seed, stream, layer, bs_, hs_)
    k1 = torch.from_numpy(k1.astype(np.int64)).to(device)[:, None]
    k2 = torch.from_numpy(k2.astype(np.int64)).to(device)[:, None]
    idx = torch.arange(start, start + count, dtype=torch.int64, device=device)[None, :]
    v = _mix32_torch(_mix32_torch(idx ^ k1) ^ k2)
    return normal_table_torch(device)[v >> 16]


class QueryStreamTorch:
    """Device twin of :class:`QueryStream`: the same bits, generated with torch ops."""

    def __init__(self, w: Workload, layer: int, device):
        import torch

        self.w, self.layer, self.device = w, layer, device
        self.step = 0
        self.bb = np.repeat(np.arange(w.B), w.Hq)
        self.hq = np.tile(np.arange(w.Hq), w.B)
        self.drift = _DriftDirs(w, layer) if w.hot_mode == "drift" else None
        if self.drift is None:
            u = np.stack([unit_dir(w, layer, b, h) for b in range(w.B) for h in range(w.Hkv)])
            u = u.reshape(w.B, w.Hkv, 1, w.d).repeat(w.G, axis=2).reshape(w.B * w.Hq, w.d).astype(np.float64)
            self.u2 = torch.from_numpy(2.0 * u).to(device)
        self.e = None
        self.a = math.sqrt(1.0 - w.rho * w.rho)

    def next(self):
        import torch

        w, d, dev = self.w, self.w.d, self.device
        if self.drift is not None:  # the drifting direction is a few host flops per head
            self.u2 = torch.from_numpy(2.0 * self.drift.next()).to(dev)
        if self.e is None:
            self.e = hash_normals_multi_torch(w.seed, STREAM_QNOISE, self.layer, self.bb, self.hq, 0, d,
                                              dev).double()
        else:
            xi = hash_normals_multi_torch(w.seed, STREAM_QNOISE, self.layer, self.bb, self.hq, self.step * d, d,
                                          dev).double()
            self.e = w.rho * self.e + self.a * xi
        qf = (self.u2 + self.e).float()
        la = hash_normals_multi_torch(w.seed, STREAM_LANOISE, self.layer, self.bb, self.hq,
                                      self.step * w.n_la * d, w.n_la * d, dev).double().view(-1, w.n_la, d)
        qla = (qf.double()[:, None, :] + w.la_sigma * la).float()
        self.step += 1
        q = qf.to(torch.bfloat16).view(w.B, w.Hq, d)
        qla = qla.to(torch.bfloat16).view(w.B, w.Hq, w.n_la, d).transpose(1, 2).contiguous()
        return q, qla
