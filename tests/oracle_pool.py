"""The oracle's layer step run head by head in a pool of worker processes.

Every (request, KV head) of a layer step is independent in the oracle, so a
large case is cut into one-head problems (B = 1, Hkv = 1 slices of every input)
that worker processes solve with ``oracle.oasis_ref.layer_step``; the results
are put back together in the layout ``layer_step`` itself returns, and the
tables and pools are updated in place exactly as the one-process call updates
them.  The pool uses the "spawn" start method, so it is safe to create after the
parent process has initialised CUDA.
"""
import multiprocessing
import os
from concurrent.futures import ProcessPoolExecutor

import numpy as np

_POOL = None


def pool():
    global _POOL
    if _POOL is None:
        n = max(1, min(16, (os.cpu_count() or 2) - 1))
        _POOL = ProcessPoolExecutor(max_workers=n, mp_context=multiprocessing.get_context("spawn"))
    return _POOL


def _one_head(args):
    from oracle import oasis_ref as ref

    K, qla, q, ctx, host, kp, vp, b2s, s2b, lu, Kb, C, step, kw = args
    r = ref.layer_step(K, qla, q, [ctx], host, kp, vp, b2s, s2b, lu, Kb, C, step, **kw)
    out = {"S": r["S"][(0, 0)], "F": r["F"][(0, 0)], "A": r["A"][(0, 0)], "copies": r["copies"][(0, 0)],
           "score": r["score"][(0, 0)], "out": r["out"][0], "b2s": b2s, "s2b": s2b, "lu": lu}
    # only the slots this step wrote travel back
    out["slots"] = [(p, kp[0, 0, p].copy(), vp[0, 0, p].copy()) for (_, p) in r["copies"][(0, 0)]]
    if "out_la" in r:
        out["out_la"] = r["out_la"][0]
    return out


def layer_step(K, qla, q, ctx, host, kp, vp, b2s, s2b, lu, Kb, C, step, heads=None, prev_S=None, **kw):
    """Same arguments, result and in-place updates as oracle.oasis_ref.layer_step,
    computed by the worker pool."""
    B, Hkv = K.shape[:2]
    G = q.shape[1] // Hkv
    pairs = heads if heads is not None else [(b, h) for b in range(B) for h in range(Hkv)]
    jobs = []
    for (b, h) in pairs:
        g = slice(h * G, (h + 1) * G)
        hk = dict(kw)
        if prev_S is not None:
            hk["prev_S"] = {(0, 0): prev_S[(b, h)]}
        jobs.append((K[b:b + 1, h:h + 1], qla[b:b + 1, :, g], q[b:b + 1, g], int(ctx[b]), host[b:b + 1, h:h + 1],
                     kp[b:b + 1, h:h + 1].copy(), vp[b:b + 1, h:h + 1].copy(), b2s[b:b + 1, h:h + 1].copy(),
                     s2b[b:b + 1, h:h + 1].copy(), lu[b:b + 1, h:h + 1].copy(), Kb, C, step, hk))
    res = {"S": {}, "F": {}, "A": {}, "copies": {}, "score": {}, "out": np.zeros((B, q.shape[1], q.shape[2]))}
    if kw.get("lookahead_out"):
        res["out_la"] = np.zeros((B, qla.shape[1], q.shape[1], q.shape[2]))
    for (b, h), r in zip(pairs, pool().map(_one_head, jobs, chunksize=max(1, len(jobs) // 64))):
        for k in ("S", "F", "A", "copies", "score"):
            res[k][(b, h)] = r[k]
        res["out"][b, h * G:(h + 1) * G] = r["out"]
        if "out_la" in r:
            res["out_la"][b, :, h * G:(h + 1) * G] = r["out_la"]
        b2s[b, h], s2b[b, h], lu[b, h] = r["b2s"][0, 0], r["s2b"][0, 0], r["lu"][0, 0]
        for (p, kk, vv) in r["slots"]:
            kp[b, h, p], vp[b, h, p] = kk, vv
    return res


def slot_digests(kp_head, vp_head, s2b_head):
    """Per occupied slot p: (p, digest of its K and V bytes) - compares pool contents
    without moving them between processes."""
    import hashlib

    out = []
    for p in range(len(s2b_head)):
        if s2b_head[p] >= 0:
            h = hashlib.blake2b(digest_size=12)
            h.update(np.ascontiguousarray(kp_head[p]).tobytes())
            h.update(np.ascontiguousarray(vp_head[p]).tobytes())
            out.append((p, h.digest()))
    return out


def head_history(spec):
    """One (layer, request, KV head) of a multi-layer workload, from its seeded
    inputs through `steps` oracle layer steps.

    spec = (w, layer, b, h, l_host, steps, scoring, lag): the host tier of layer
    l is host buffer l mod l_host, which holds the keys and values of layer
    l mod l_host (the engine's aliasing of host layers); the key cache and the
    initially resident slots hold layer l's own data.  ``lag``: the cross-step
    order (attention over the previous step's selection from step 1 on).
    Returns per step: S, F, out [G][d], the head's tables and pool digests.
    """
    from oracle import oasis_ref as ref
    from sparse_decode_attention_oasis_gb300 import synthetic as syn

    w, l, b, h, l_host, steps, scoring, lag = spec
    K, V = syn.head_kv(w, l, b, h)
    lh = l % l_host
    Kh, Vh = (K, V) if lh == l else syn.head_kv(w, lh, b, h)
    sub = syn.Workload("sub", L=1, B=1, Hq=w.G, Hkv=1, ctx=[w.ctx[b]], Kb=w.Kb, C=w.C, n_la=w.n_la,
                       nb_max=w.nb_max, P=w.P)
    host = syn.host_tier_from_kv(sub, Kh[None, None], Vh[None, None])
    own = syn.host_tier_from_kv(sub, K[None, None], V[None, None])
    b2s, s2b, lu = [t[b:b + 1, h:h + 1].copy() for t in syn.initial_tables(w, l)]
    kp, vp = syn.pools_from_tables(sub, own, s2b)
    hist, prev = [], None
    for s in range(steps):
        q, qla = syn.head_queries(w, l, b, h, s)
        r = ref.layer_step(K[None, None], qla[None], q[None], [w.ctx[b]], host, kp, vp, b2s, s2b, lu,
                           w.Kb, w.C, s, scoring=scoring, prev_S=prev)
        if lag:
            prev = {(0, 0): r["S"][(0, 0)]}
        hist.append({"S": r["S"][(0, 0)], "F": r["F"][(0, 0)], "out": r["out"][0], "b2s": b2s[0, 0].copy(),
                     "s2b": s2b[0, 0].copy(), "lu": lu[0, 0].copy(),
                     "pool": slot_digests(kp[0, 0], vp[0, 0], s2b[0, 0])})
    return hist


def head_histories(specs):
    """head_history for every spec, in the worker pool (results in spec order)."""
    return list(pool().map(head_history, specs))
