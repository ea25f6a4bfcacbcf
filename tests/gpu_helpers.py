"""Shared pieces of the GPU parity tests: one layer held on the GPU and in oracle arrays."""
import numpy as np

from oracle import oasis_ref as ref
from sparse_decode_attention_oasis_gb300 import synthetic as syn

ATOL, RTOL = 2e-3, 1e-2


def _dev_bits(bits):
    import torch

    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def _check_out(got, want, what=""):
    err = np.abs(got - want)
    ok = (err <= ATOL) | (err <= RTOL * np.abs(want))
    assert ok.all(), f"{what}: {int((~ok).sum())} elements out of tolerance, max abs {err.max():.3e}"
    return float(err.max())


class Case:
    """One layer of a workload held both on the GPU and in oracle arrays."""

    def __init__(self, w, K=None, V=None, tables=None, scoring="maxdot"):
        from sparse_decode_attention_oasis_gb300.engine import DecodeState

        self.w = w
        if K is None:
            K, V = syn.layer_kv(w, 0)
        self.K, self.V = K, V
        self.host = syn.host_tier_from_kv(w, K, V)
        if tables is None:
            tables = syn.initial_tables(w, 0)
        self.b2s, self.s2b, self.lu = [np.array(t) for t in tables]
        self.kp, self.vp = syn.pools_from_tables(w, self.host, self.s2b)
        self.scoring = scoring
        self.st = DecodeState(w, l_phys=1, scoring=scoring)
        self.st.fill_layer_numpy(0, K, V, self.b2s, self.s2b, self.lu)

    def step(self, step, q=None, qla=None, C=None, append=False, gather="fused", lookahead=False):
        import torch

        w = self.w
        if append:
            kn, vn = syn.append_tokens(w, 0, step)
            ref.append_token(self.K, self.host, self.kp, self.vp, self.b2s, w.ctx, kn, vn, bs=w.bs)
            for b in range(w.B):
                self.V[b, :, w.ctx[b] - 1] = vn[b]
            self.st.append_tokens(0, _dev_bits(kn), _dev_bits(vn), advance=True)
        if q is None:
            q, qla = syn.layer_queries(w, 0, step)
        if C is not None:
            w.C = C
        if w.B * w.Hkv >= 8 and w.nb_max >= 1024:  # large case: the oracle head by head in worker processes
            import oracle_pool

            r = oracle_pool.layer_step(self.K, qla, q, w.ctx, self.host, self.kp, self.vp, self.b2s, self.s2b,
                                       self.lu, w.Kb, w.C, step, scoring=self.scoring, lookahead_out=lookahead)
        else:
            r = ref.layer_step(self.K, qla, q, w.ctx, self.host, self.kp, self.vp, self.b2s, self.s2b,
                               self.lu, w.Kb, w.C, step, bs=w.bs, scoring=self.scoring, lookahead_out=lookahead)
        sc = self.st.layer_step(0, _dev_bits(qla), _dev_bits(q), step, gather=gather)
        torch.cuda.synchronize()
        self.compare(r, sc)
        if lookahead:
            out = torch.empty((w.B, w.Hq, w.d), dtype=torch.float32, device="cuda")
            out_la = torch.empty((w.B, w.n_la, w.Hq, w.d), dtype=torch.float32, device="cuda")
            self.st.attend_lookahead(0, _dev_bits(q), _dev_bits(qla), sc, out, out_la)
            torch.cuda.synchronize()
            _check_out(out.cpu().numpy().astype(np.float64), r["out"], "fused true-query rows")
            _check_out(out_la.cpu().numpy().astype(np.float64), r["out_la"], "fused lookahead rows")
        return r, sc

    def compare(self, r, sc):
        import torch

        w = self.w
        scores = sc.scores.cpu().numpy()
        sel = sc.sel.cpu().numpy()
        nsel = sc.nsel.cpu().numpy()
        fetch = sc.fetch.cpu().numpy()
        nfetch = sc.nfetch.cpu().numpy()
        assert int(sc.err.cpu()[0]) == 0
        for (b, h), S in r["S"].items():
            nb = w.nb(b)
            s_exact, _ = r["score"][(b, h)]
            if nb > w.Kb:  # scores are only needed (and written) when there is a choice
                approx = scores[b, h, :nb, 0].astype(np.float64)
                bound = scores[b, h, :nb, 1].astype(np.float64)
                assert (np.abs(approx - s_exact) <= bound).all(), f"score outside bound at {(b, h)}"
                assert (bound < 1e-2 * (1 + np.abs(s_exact))).all()
            assert nsel[b, h] == len(S)
            assert sel[b, h, :len(S)].tolist() == S, f"sel mismatch at {(b, h)}"
            assert (sel[b, h, len(S):] == -1).all()
            F = r["F"][(b, h)]
            assert nfetch[b, h] == len(F)
            assert fetch[b, h, :len(F)].tolist() == F, f"fetch mismatch at {(b, h)}"
        lp = 0
        np.testing.assert_array_equal(self.st.blk2slot[lp].cpu().numpy(), self.b2s)
        np.testing.assert_array_equal(self.st.slot2blk[lp].cpu().numpy(), self.s2b)
        np.testing.assert_array_equal(self.st.last_used[lp].cpu().numpy(), self.lu)
        kpool = self.st.k_pool[lp].cpu().view(torch.int16).numpy().view(np.uint16)
        vpool = self.st.v_pool[lp].cpu().view(torch.int16).numpy().view(np.uint16)
        occupied = self.s2b >= 0
        np.testing.assert_array_equal(kpool[occupied], self.kp[occupied])
        np.testing.assert_array_equal(vpool[occupied], self.vp[occupied])
        _check_out(sc.out.cpu().numpy().astype(np.float64), r["out"], "attention")



    def compare_pooled(self):
        """Pooled keys on the GPU against the oracle's pooling of the current keys (values)."""
        import torch

        w = self.w
        got = self.st.Kp[0].float().cpu().numpy()
        for b in range(w.B):
            for h in range(w.Hkv):
                hi, lo = ref.pool_keys(self.K[b, h], w.ctx[b], w.nb_max, w.bs)
                np.testing.assert_array_equal(got[b, h, :, 0], ref.bf16_to_f64(hi))
                np.testing.assert_array_equal(got[b, h, :, 1], ref.bf16_to_f64(lo))

    def compare_caches(self):
        """Keys in HBM and the whole host tier, bit for bit."""
        import torch

        kh = self.st.K[0].cpu().view(torch.int16).numpy().view(np.uint16)
        np.testing.assert_array_equal(kh, self.K)
        host = self.st.host[0].view(torch.int16).numpy().view(np.uint16)
        np.testing.assert_array_equal(host, self.host)
        np.testing.assert_array_equal(self.st.ctx.cpu().numpy(), np.array(self.w.ctx))
