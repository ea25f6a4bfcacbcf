"""Plain CPU oracle for the OasisKV lookahead sparse decode step (float64 / exact).

TEST INFRASTRUCTURE ONLY.  This module is the checker the CUDA path is compared
against.  Only the test-suite, the package smoke check and the benchmark's CPU
baseline leg may import or call it; the library itself never does, and it shares
no code with the CUDA kernels (it takes plain numpy arrays of bfloat16 bit
patterns and int32 tables).

Sources (the pages about "OasisKV: Scaling In-Decode KV Cache Beyond HBM with
Lookahead Sparse Prefetching"):
  [abs]   the paper abstract (chatpaper.ai and newx.sg pages, "Abstract"):
          keep only the most relevant tokens' KV in HBM, predict them with
          lookahead (speculative-decoding draft) tokens, prefetch them from a
          host tier, 2,048-token KV budget.
  [steps] metalmedia.ai page, explanatory figure, steps 2-4: the lookahead
          prediction of next-step KV blocks; comparing the prediction with the
          blocks already on the GPU and fetching only the missing ones, under a
          per-step cap; the predict/select/transfer pipeline.
  [fig7]  metalmedia.ai page, Figure 7 caption (look-ahead attention): the
          draft queries are compared with the keys to pick the K blocks the next
          decode step will need; attention itself only reads the sparse set of
          blocks kept on the GPU.
  [fig9]  metalmedia.ai page, Figure 9 caption: a head-wise table maps each GPU
          block of the bounded working set to a CPU (host-tier) block.
  [tab2]  metalmedia.ai page, Table 2 caption: a fetch ratio sets how many
          blocks a single step may bring in; evictions follow LRU.
  [fig6]  metalmedia.ai page, Figure 6 caption: per layer, how well the top-K
          set predicted by the draft query agrees with the exact top-K set of
          the true next-token query.
  [fig4]  metalmedia.ai page, Figure 4 caption: top-20 block prediction
          accuracy per layer from the previous token versus a lookahead token.
  [fig8]  metalmedia.ai page, Figure 8 caption: across two decode steps, the
          draft query of step t drives a layer's top-K prediction, selection and
          transfer, which complete before that layer's attention at step t+1.

Readings where the pages are silent (each is listed in the design notes):
  * score(b) = max over lookahead queries j, query heads g of the GQA group of
    KV head h, and valid tokens t of block b, of q_la[j, hG+g] . k_t / sqrt(d)
    (the exact real value; the pages' min/max pooled summary is not used).
  * ranking: larger exact score first; equal exact scores -> lower block index.
  * the selected set S and the fetch list F are sets; they are emitted in
    ascending block order, and F[i] (ascending) is paired with the i-th
    candidate slot (free slots ascending, then LRU victims).
  * LRU victims are resident blocks not in S, ordered by (last_used, block);
    last_used is the last step a block was attended; initial residents have -1.
  * attention runs over A = S intersected with the resident set after the
    gather, on valid tokens t < ctx only; if A is empty the output is zero.

Exactness: every bfloat16 value is an integer multiple of 2**-133, so every
product q_i*k_i is exact in float64 and every dot product is an integer
multiple of 2**-266.  ``head_block_scores`` evaluates dot products with a
float64 matrix product only where a per-dot test proves the float64 sum exact
(all partial sums are multiples of 2**L and bounded by 2**(L+52)); any other
dot is evaluated with Python integers.  Ranking keys are therefore exact.
"""
from __future__ import annotations

import math
from typing import Dict, List, Sequence, Tuple

import numpy as np

BS_DEFAULT = 16
_EXACT_SHIFT = 133  # bf16 value * 2**133 is an integer


# --------------------------------------------------------------------------
# bfloat16 helpers
# --------------------------------------------------------------------------
def bf16_to_f64(bits) -> np.ndarray:
    """bfloat16 bit patterns -> float64 (exact)."""
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


def _lsb_lower_bound(x: np.ndarray) -> np.ndarray:
    """Lower bound on log2 of the least significant set bit of each bf16 value.

    A bf16 value with frexp exponent e is a multiple of 2**(e-8); zero gets a
    huge sentinel so that it never tightens a minimum.
    """
    _, e = np.frexp(x)
    out = e.astype(np.int64) - 8
    out[x == 0] = 1 << 20
    return out


def _to_int(x: np.ndarray) -> List[int]:
    return [int(v) for v in np.ldexp(x, _EXACT_SHIFT)]


# --------------------------------------------------------------------------
# a1: block scores  ([fig7], [steps] step 2)
# --------------------------------------------------------------------------
def head_block_scores(K: np.ndarray, Q: np.ndarray, ctx: int, bs: int = BS_DEFAULT):
    """Exact block scores of one KV head.

    K: float64 [T][d] (exact bf16 values), Q: float64 [N][d] (the n_la*G
    lookahead queries of the head), ctx: valid tokens.  Returns
    ``(score, key)``: ``score`` float64 [nb] = max_{t in blk, t<ctx, n} Q[n].K[t]
    (unscaled, i.e. sqrt(d) times the block score), rounded to nearest when it is
    not exactly representable; ``key`` a list of exact integers equal to
    score * 2**266, used for all comparisons.
    """
    nb = -(-ctx // bs)
    Kv = K[:ctx]
    D = Kv @ Q.T                                  # [ctx][N]
    A = np.abs(Kv) @ np.abs(Q).T                  # sum of |products|
    Lk = _lsb_lower_bound(Kv).min(axis=1)
    Lq = _lsb_lower_bound(Q).min(axis=1)
    L = Lk[:, None] + Lq[None, :]
    with np.errstate(over="ignore"):
        ok = A < np.ldexp(1.0, np.minimum(L + 52, 2000))
    pad = nb * bs - ctx
    if ok.all():
        Dp = np.concatenate([D, np.full((pad, D.shape[1]), -np.inf)]) if pad else D
        score = Dp.reshape(nb, bs * D.shape[1]).max(axis=1)
        key = [int(v) for v in np.ldexp(score, 2 * _EXACT_SHIFT)]
        return score, key
    # slow exact path for the dots the float64 test could not certify
    Kq = [_to_int(row) for row in Kv]
    Qq = [_to_int(row) for row in Q]
    key = []
    for blk in range(nb):
        best = None
        for t in range(blk * bs, min(ctx, (blk + 1) * bs)):
            for n in range(Q.shape[0]):
                if ok[t, n]:
                    v = int(np.ldexp(D[t, n], 2 * _EXACT_SHIFT))
                else:
                    v = sum(a * b for a, b in zip(Kq[t], Qq[n]))
                if best is None or v > best:
                    best = v
        key.append(best)
    score = np.array([math.ldexp(float(k), -2 * _EXACT_SHIFT) if abs(k) < 2 ** 1000
                      else float(k) * 2.0 ** (-2 * _EXACT_SHIFT) for k in key])
    return score, key


def head_queries_f64(q_la_bits: np.ndarray, b: int, h: int, G: int) -> np.ndarray:
    """The n_la*G lookahead query rows of KV head h: q_la[b, j, h*G + g], ordered (j, g)."""
    q = bf16_to_f64(q_la_bits[b, :, h * G:(h + 1) * G, :])     # [n_la][G][d]
    return q.reshape(-1, q.shape[-1])


def block_scores(k_bits: np.ndarray, q_la_bits: np.ndarray, ctx_len: Sequence[int],
                 bs: int = BS_DEFAULT, heads=None):
    """Scores of every block of every (request, KV head) of one layer.

    k_bits: bf16 [B][Hkv][T_max][d]; q_la_bits: bf16 [B][n_la][Hq][d].
    Returns dict (b, h) -> (score_scaled float64 [nb], exact key list); the
    scaled score includes the 1/sqrt(d) factor of the definition.
    """
    B, Hkv, _, d = k_bits.shape
    Hq = q_la_bits.shape[2]
    G = Hq // Hkv
    out = {}
    pairs = heads if heads is not None else [(b, h) for b in range(B) for h in range(Hkv)]
    for (b, h) in pairs:
        K = bf16_to_f64(k_bits[b, h])
        Q = head_queries_f64(q_la_bits, b, h, G)
        score, key = head_block_scores(K, Q, int(ctx_len[b]), bs)
        out[(b, h)] = (score / math.sqrt(d), key)
    return out


# --------------------------------------------------------------------------
# f1: block scores from min/max pooled compressed keys  ([fig7] left)
# --------------------------------------------------------------------------
def pool_keys(k_bits: np.ndarray, ctx: int, nb_max: int, bs: int = BS_DEFAULT):
    """Per-block min/max pooling of one head's keys.

    k_bits: bf16 [T_max][d].  Returns (hi, lo) bf16 bit arrays [nb_max][d]:
    hi[x][i] = max over the valid tokens t of block x (t < ctx) of k[t][i], lo
    the minimum; blocks without a valid token are all zero.  A maximum of bf16
    values is one of them, so the pooled keys are exact bf16.
    """
    T, d = k_bits.shape
    hi = np.zeros((nb_max, d), np.uint16)
    lo = np.zeros((nb_max, d), np.uint16)
    vals = bf16_to_f64(k_bits)
    for x in range(min(nb_max, -(-ctx // bs))):
        rows = list(range(x * bs, min(ctx, (x + 1) * bs)))
        v = vals[rows]
        ih = v.argmax(axis=0)
        il = v.argmin(axis=0)
        hi[x] = k_bits[[rows[j] for j in ih], range(d)]
        lo[x] = k_bits[[rows[j] for j in il], range(d)]
    return hi, lo


def head_block_scores_pooled(hi_bits: np.ndarray, lo_bits: np.ndarray, Q: np.ndarray, nb: int):
    """Exact pooled block scores of one KV head.

    hi_bits, lo_bits: bf16 [nb_max][d] from pool_keys; Q: float64 [N][d] (the head's
    lookahead query rows).  For block x:
        pooled(x) = max over n of  sum_i max(Q[n][i] * hi[x][i], Q[n][i] * lo[x][i])
    (unscaled), i.e. for each query the largest value any key inside the block's
    per-dimension [lo, hi] box can reach, an upper bound of the block's max-dot
    score.  Returns (score float64 [nb], exact integer keys = pooled x 2^266).
    """
    H = bf16_to_f64(hi_bits[:nb])
    Lo = bf16_to_f64(lo_bits[:nb])
    terms = np.maximum(H[:, None, :] * Q[None, :, :], Lo[:, None, :] * Q[None, :, :])  # [nb][N][d]
    D = terms.sum(axis=2)
    A = np.abs(terms).sum(axis=2)
    Lk = np.minimum(_lsb_lower_bound(H).min(axis=1), _lsb_lower_bound(Lo).min(axis=1))
    Lq = _lsb_lower_bound(Q).min(axis=1)
    L = Lk[:, None] + Lq[None, :]
    with np.errstate(over="ignore"):
        ok = A < np.ldexp(1.0, np.minimum(L + 52, 2000))
    if ok.all():
        score = D.max(axis=1)
        return score, [int(v) for v in np.ldexp(score, 2 * _EXACT_SHIFT)]
    Hq = [_to_int(r) for r in H]
    Lq_ = [_to_int(r) for r in Lo]
    Qq = [_to_int(r) for r in Q]
    key = []
    for x in range(nb):
        best = None
        for n in range(Q.shape[0]):
            if ok[x, n]:
                v = int(np.ldexp(D[x, n], 2 * _EXACT_SHIFT))
            else:
                v = sum(max(q * a, q * b) for q, a, b in zip(Qq[n], Hq[x], Lq_[x]))
            best = v if best is None or v > best else best
        key.append(best)
    score = np.array([math.ldexp(float(k), -2 * _EXACT_SHIFT) if abs(k) < 2 ** 1000
                      else float(k) * 2.0 ** (-2 * _EXACT_SHIFT) for k in key])
    return score, key


def block_scores_pooled(pooled: Dict, q_la_bits: np.ndarray, ctx_len: Sequence[int], d: int,
                        bs: int = BS_DEFAULT, heads=None):
    """Pooled scores of every (request, KV head): pooled[(b, h)] = (hi, lo) bits.

    Returns dict (b, h) -> (score scaled by 1/sqrt(d), exact key list), like
    block_scores.
    """
    Hq = q_la_bits.shape[2]
    Hkv = len({h for (_, h) in pooled})
    G = Hq // Hkv
    out = {}
    for (b, h) in (heads if heads is not None else sorted(pooled)):
        hi, lo = pooled[(b, h)]
        Q = head_queries_f64(q_la_bits, b, h, G)
        nb = -(-int(ctx_len[b]) // bs)
        score, key = head_block_scores_pooled(hi, lo, Q, nb)
        out[(b, h)] = (score / math.sqrt(d), key)
    return out


# --------------------------------------------------------------------------
# a2: top-K under the token budget  ([abs] 2,048-token budget, [fig7] top-K)
# --------------------------------------------------------------------------
def rank_order(key: Sequence[int], blocks: Sequence[int]) -> List[int]:
    """Blocks sorted by (exact score descending, block index ascending)."""
    return sorted(blocks, key=lambda x: (-key[x], x))


def topk_select(key: Sequence[int], Kb: int) -> List[int]:
    """S = the min(Kb, nb) highest-ranked blocks, returned in ascending block order."""
    nb = len(key)
    top = rank_order(key, range(nb))[: min(Kb, nb)]
    return sorted(top)


# --------------------------------------------------------------------------
# a3: diff against the resident set, capped  ([steps] step 3, [tab2])
# --------------------------------------------------------------------------
def fetch_diff_capped(S: Sequence[int], blk2slot: np.ndarray, C: int,
                      key: Sequence[int]) -> List[int]:
    """F = the min(C, |M|) highest-ranked blocks of M = {x in S : x not resident}.

    Returned in ascending block order.
    """
    M = [x for x in S if blk2slot[x] < 0]
    top = rank_order(key, M)[: max(0, min(C, len(M)))]
    return sorted(top)


# --------------------------------------------------------------------------
# a4: slot assignment, host -> HBM copy, table update  ([fig9], [tab2], [steps] 4)
# --------------------------------------------------------------------------
def assign_slots(S: Sequence[int], F: Sequence[int], blk2slot: np.ndarray,
                 slot2blk: np.ndarray, last_used: np.ndarray, step: int):
    """Update one head's tables in place; return the copies [(block, slot)].

    Candidate slots: free slots in ascending order, then LRU victims = resident
    blocks outside S ordered by (last_used, block).  F[i] (ascending) takes the
    i-th candidate.  Afterwards every block of A = S intersect resident gets
    last_used = step.
    """
    Sset = set(int(x) for x in S)
    P = slot2blk.shape[0]
    free = [p for p in range(P) if slot2blk[p] < 0]
    victims = [p for p in range(P) if slot2blk[p] >= 0 and int(slot2blk[p]) not in Sset]
    victims.sort(key=lambda p: (int(last_used[p]), int(slot2blk[p])))
    cand = free + victims
    if len(F) > len(cand):
        raise ValueError("not enough slots for the fetch list")
    copies = []
    for i, x in enumerate(sorted(F)):
        p = cand[i]
        old = int(slot2blk[p])
        if old >= 0:
            blk2slot[old] = -1
        blk2slot[x] = p
        slot2blk[p] = x
        copies.append((int(x), int(p)))
    for x in S:
        p = int(blk2slot[x])
        if p >= 0:
            last_used[p] = step
    return copies


def attended_blocks(S: Sequence[int], blk2slot: np.ndarray) -> List[int]:
    """A = blocks of S that are resident after the gather (ascending)."""
    return [int(x) for x in sorted(S) if blk2slot[x] >= 0]


# --------------------------------------------------------------------------
# a5: sparse decode attention  ([fig7] right, [abs])
# --------------------------------------------------------------------------
def attention_over_tokens(q: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float) -> np.ndarray:
    """softmax(scale * q K^T) V for q [G][d], K/V [T][d] (float64); T = 0 gives zeros."""
    if K.shape[0] == 0:
        return np.zeros((q.shape[0], V.shape[1]))
    logits = scale * (q @ K.T)
    m = logits.max(axis=1, keepdims=True)
    p = np.exp(logits - m)
    return (p @ V) / p.sum(axis=1, keepdims=True)


def head_sparse_attention(q_bits: np.ndarray, kpool_bits: np.ndarray, vpool_bits: np.ndarray,
                          A: Sequence[int], blk2slot: np.ndarray, ctx: int, scale: float,
                          bs: int = BS_DEFAULT) -> np.ndarray:
    """Attention of one KV head's G true queries over the valid tokens of A.

    q_bits [G][d]; kpool/vpool bits [P][bs][d] (this head's HBM slots).
    """
    rows_k, rows_v = [], []
    for x in sorted(A):
        p = int(blk2slot[x])
        n = min(bs, ctx - x * bs)
        rows_k.append(kpool_bits[p, :n])
        rows_v.append(vpool_bits[p, :n])
    d = q_bits.shape[-1]
    K = bf16_to_f64(np.concatenate(rows_k)) if rows_k else np.zeros((0, d))
    V = bf16_to_f64(np.concatenate(rows_v)) if rows_v else np.zeros((0, d))
    return attention_over_tokens(bf16_to_f64(q_bits), K, V, scale)


# --------------------------------------------------------------------------
# token append (long-output decode)  ([abs]: the KV cache grows during decode)
# --------------------------------------------------------------------------
def append_token(k_bits, host_kv, k_pool, v_pool, blk2slot, ctx_len, k_new, v_new,
                 bs: int = BS_DEFAULT, advance: bool = True):
    """Append one token per request to keys, host tier and (if resident) its slot.

    k_bits [B][Hkv][T_max][d]; host_kv [B][Hkv][nb_max][2][bs][d];
    k_pool/v_pool [B][Hkv][P][bs][d]; blk2slot [B][Hkv][nb_max]; ctx_len is a
    mutable list/array of per-request lengths; k_new/v_new [B][Hkv][d].  With
    ``advance`` the lengths grow by one (a model calls this once per layer and
    advances on the last).  A full cache leaves the request unchanged.
    """
    B, Hkv, T_max, _ = k_bits.shape
    for b in range(B):
        t = int(ctx_len[b])
        if t < 0 or t >= T_max:
            continue
        blk, r = divmod(t, bs)
        for h in range(Hkv):
            k_bits[b, h, t] = k_new[b, h]
            host_kv[b, h, blk, 0, r] = k_new[b, h]
            host_kv[b, h, blk, 1, r] = v_new[b, h]
            p = int(blk2slot[b, h, blk])
            if p >= 0:
                k_pool[b, h, p, r] = k_new[b, h]
                v_pool[b, h, p, r] = v_new[b, h]
        if advance:
            ctx_len[b] = t + 1


# --------------------------------------------------------------------------
# f3: agreement of a predicted top-K set with the exact one  ([fig6], [fig4])
# --------------------------------------------------------------------------
def exact_topk_true_query(k_bits: np.ndarray, q_bits: np.ndarray, ctx_len: Sequence[int], Kb: int,
                          bs: int = BS_DEFAULT, heads=None) -> Dict:
    """Per head, the top-Kb set of the true next-token query.

    The same block score as a1 with the true queries of the GQA group in place of
    the lookahead ones (one "lookahead" position): the exact set against which
    Figure 6 measures the draft query's prediction.
    """
    q1 = q_bits[:, None]  # [B][1][Hq][d]
    scores = block_scores(k_bits, q1, ctx_len, bs, heads=heads)
    return {bh: topk_select(key, Kb) for bh, (_, key) in scores.items()}


def set_agreement(pred: Sequence[int], exact: Sequence[int], blk2slot: np.ndarray = None):
    """(|pred & exact|, |pred & exact & resident|, |exact|) for one head.

    The first count over |exact| is the per-head agreement of Figure 6 (and, at
    K = 20 with the previous token's query as the predictor, of Figure 4); the
    second counts the exact blocks that attention actually reads when pred is
    the selected set (resident = blk2slot >= 0 after the gather).
    """
    common = set(int(x) for x in pred) & set(int(x) for x in exact)
    res = sum(1 for x in common if blk2slot is not None and blk2slot[x] >= 0)
    return len(common), res, len(set(int(x) for x in exact))


# --------------------------------------------------------------------------
# one layer-step over a whole batch (a1 -> a5)
# --------------------------------------------------------------------------
def layer_step(k_bits, q_la_bits, q_bits, ctx_len, host_kv, k_pool, v_pool,
               blk2slot, slot2blk, last_used, Kb: int, C: int, step: int,
               scale: float = None, bs: int = BS_DEFAULT, heads=None, scoring: str = "maxdot",
               prev_S: Dict = None, lookahead_out: bool = False) -> Dict:
    """Run a1..a5 for one layer.  Tables and pools are updated in place.

    host_kv bits [B][Hkv][nb_max][2][bs][d]; k_pool/v_pool bits [B][Hkv][P][bs][d].
    scoring: "maxdot" (a1, the exact max over tokens) or "pooled" (f1, the score
    from the per-block min/max pooled keys of the valid tokens).
    prev_S: the cross-step pipeline of [fig8] (f4): the lookahead queries of the
    previous step chose this step's blocks.  Attention then runs first, over
    A = prev_S[(b, h)] intersected with the blocks resident on entry (the previous
    step's gather brought them in), with the pools as they are on entry; the
    selection and gather of this step only prepare the next one.
    lookahead_out: also attend the lookahead queries over the same A (f2, the
    fused look-ahead attention of [fig7] right): res["out_la"] [B][n_la][Hq][d].
    Returns dict with per-head S, F, copies, A and out float64 [B][Hq][d].
    """
    B, Hkv, T_max, d = k_bits.shape
    Hq = q_bits.shape[1]
    G = Hq // Hkv
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    pairs = heads if heads is not None else [(b, h) for b in range(B) for h in range(Hkv)]
    if scoring == "pooled":
        nb_max = T_max // bs
        pooled = {(b, h): pool_keys(k_bits[b, h], int(ctx_len[b]), nb_max, bs) for (b, h) in pairs}
        scores = block_scores_pooled(pooled, q_la_bits, ctx_len, d, bs, heads=pairs)
    elif scoring == "maxdot":
        scores = block_scores(k_bits, q_la_bits, ctx_len, bs, heads=pairs)
    else:
        raise ValueError(scoring)
    n_la = q_la_bits.shape[1]
    res = {"S": {}, "F": {}, "copies": {}, "A": {}, "score": {},
           "out": np.zeros((B, Hq, d))}
    if lookahead_out:
        res["out_la"] = np.zeros((B, n_la, Hq, d))

    def attend_la(b, h, A):
        if lookahead_out:
            for j in range(n_la):
                res["out_la"][b, j, h * G:(h + 1) * G] = head_sparse_attention(
                    q_la_bits[b, j, h * G:(h + 1) * G], k_pool[b, h], v_pool[b, h], A, blk2slot[b, h],
                    int(ctx_len[b]), scale, bs)
    if prev_S is not None:
        for (b, h) in pairs:
            A = attended_blocks(prev_S[(b, h)], blk2slot[b, h])
            res["out"][b, h * G:(h + 1) * G] = head_sparse_attention(
                q_bits[b, h * G:(h + 1) * G], k_pool[b, h], v_pool[b, h], A, blk2slot[b, h], int(ctx_len[b]),
                scale, bs)
            attend_la(b, h, A)
            res["A"][(b, h)] = A
    for (b, h) in pairs:
        sc, key = scores[(b, h)]
        S = topk_select(key, Kb)
        F = fetch_diff_capped(S, blk2slot[b, h], C, key)
        copies = assign_slots(S, F, blk2slot[b, h], slot2blk[b, h], last_used[b, h], step)
        for (x, p) in copies:
            k_pool[b, h, p] = host_kv[b, h, x, 0]
            v_pool[b, h, p] = host_kv[b, h, x, 1]
        if prev_S is None:
            A = attended_blocks(S, blk2slot[b, h])
            o = head_sparse_attention(q_bits[b, h * G:(h + 1) * G], k_pool[b, h], v_pool[b, h],
                                      A, blk2slot[b, h], int(ctx_len[b]), scale, bs)
            res["out"][b, h * G:(h + 1) * G] = o
            attend_la(b, h, A)
            res["A"][(b, h)] = A
        res["S"][(b, h)] = S
        res["F"][(b, h)] = F
        res["copies"][(b, h)] = copies
        res["score"][(b, h)] = (sc, key)
    return res
