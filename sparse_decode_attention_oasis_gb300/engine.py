"""Device state of a decode workload and the per-layer call sequence.

PyTorch is used only to own memory (HBM tensors, page-locked host tier) and
streams; every step of the path runs in liboasis.so through :mod:`binding`.

Layout in HBM (one physical layer buffer per entry of the first axis):
  K        bf16 [L][B][Hkv][nb_max*16][128]   keys kept in HBM for scoring
  k_pool   bf16 [L][B][Hkv][P][16][128]       HBM slots (bounded working set)
  v_pool   bf16 [L][B][Hkv][P][16][128]
  blk2slot int32 [L][B][Hkv][nb_max]          slot of a resident block or -1
  slot2blk int32 [L][B][Hkv][P]               block held by a slot or -1
  last_used int32 [L][B][Hkv][P]              LRU clock
  Kp       bf16 [L][B][Hkv][nb_max][2][128]   min/max pooled keys (pooled scoring only)
Host tier (page-locked, device-mapped): bf16 [L_host][B][Hkv][nb_max][2][16][128],
from cudaHostAlloc (default) or a huge-page mapping registered with CUDA.
Scratch sets (scores, sel, fetch, workspace, ...) alternate between consecutive
layers of a step.  When the physical layer count is smaller than the logical
one, layer l uses buffer l mod L_phys (host tier: l mod L_host).

decode_step issues a whole decode step in one of several launch orders (see its
docstring); StepGraph captures decode steps as one CUDA graph.
"""
from __future__ import annotations

import math
from typing import Optional

import numpy as np
import torch

from . import binding as B
from . import synthetic as syn


class HugePinnedBuffer:
    """Page-locked, device-mapped host memory backed by transparent huge pages.

    The host tier is read by zero-copy loads at random block positions; on a
    64 KiB-page host every block touches a different page.  An anonymous mapping
    advised MADV_HUGEPAGE (512 MiB pages) and then registered with
    cudaHostRegister(Mapped) keeps the number of translations per layer small
    (a lower gather median), but on some systems large registrations of this
    kind stalled zero-copy reads for milliseconds; DecodeState takes its host
    tier from cudaHostAlloc unless asked for this.  The memory starts zeroed.
    """

    _ALIGN = 1 << 29

    def __init__(self, nbytes: int):
        import ctypes

        libc = ctypes.CDLL("libc.so.6", use_errno=True)
        libc.mmap.restype = ctypes.c_void_p
        libc.mmap.argtypes = [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                              ctypes.c_long]
        libc.madvise.argtypes = [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int]
        libc.munmap.argtypes = [ctypes.c_void_p, ctypes.c_size_t]
        self.libc = libc
        self.map_bytes = nbytes + self._ALIGN
        raw = libc.mmap(None, self.map_bytes, 0x1 | 0x2, 0x02 | 0x20, -1, 0)  # RW, private anonymous
        if raw in (None, ctypes.c_void_p(-1).value):
            raise RuntimeError("mmap of the host tier failed")
        self.raw = raw
        self.base = (raw + self._ALIGN - 1) // self._ALIGN * self._ALIGN
        libc.madvise(ctypes.c_void_p(self.base), nbytes, 14)  # MADV_HUGEPAGE (advice only)
        rc = torch.cuda.cudart().cudaHostRegister(self.base, nbytes, 0x1 | 0x2)  # portable | mapped
        rc = int(rc[0] if isinstance(rc, tuple) else rc)
        if rc != 0:
            libc.munmap(ctypes.c_void_p(self.raw), self.map_bytes)
            raise RuntimeError(f"cudaHostRegister of the host tier failed ({rc})")
        self.nbytes = nbytes
        buf = (ctypes.c_uint8 * nbytes).from_address(self.base)
        self.tensor = torch.from_numpy(np.frombuffer(buf, dtype=np.uint8))

    def close(self):
        if getattr(self, "raw", None):
            import ctypes

            torch.cuda.cudart().cudaHostUnregister(self.base)
            self.libc.munmap(ctypes.c_void_p(self.raw), self.map_bytes)
            self.raw = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def _bf16_from_bits(bits: np.ndarray, device) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


class LayerScratch:
    """Buffers one layer-step writes: scores, selection, fetch list, output."""

    def __init__(self, shape: B.Shape, device):
        s = shape
        self.shape = s
        dev = device
        self.scores = torch.empty((s.B, s.Hkv, s.nb_max, 2), dtype=torch.float32, device=dev)
        self.sel = torch.empty((s.B, s.Hkv, s.Kb), dtype=torch.int32, device=dev)
        self.nsel = torch.empty((s.B, s.Hkv), dtype=torch.int32, device=dev)
        self.fetch = torch.empty((s.B, s.Hkv, s.Kb), dtype=torch.int32, device=dev)
        self.nfetch = torch.empty((s.B, s.Hkv), dtype=torch.int32, device=dev)
        self.ws_bytes = B.oasis_attn_workspace_bytes(s)
        self.ws = torch.empty(max(16, self.ws_bytes), dtype=torch.uint8, device=dev)
        self.out = torch.empty((s.B, s.Hq, 128), dtype=torch.float32, device=dev)
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)
        self.work = torch.zeros(2, dtype=torch.int32, device=dev)  # chunk counter of the dynamic scorer


class _SelView:
    """A scratch set whose selection (sel, nsel) lives in per-layer buffers that
    outlast the step (the cross-step pipeline reads them one step later)."""

    def __init__(self, base: LayerScratch, sel: torch.Tensor, nsel: torch.Tensor):
        self._base = base
        self.sel = sel
        self.nsel = nsel

    def __getattr__(self, name):
        return getattr(self._base, name)


class DecodeState:
    def __init__(self, w: syn.Workload, device="cuda", l_phys: Optional[int] = None,
                 l_host: Optional[int] = None, pin_host: bool = True, scoring: str = "maxdot",
                 host_alloc: str = "cuda"):
        """scoring: "maxdot" (a1, scan of the full keys) or "pooled" (f1, scan of the
        min/max pooled keys ``Kp``, bf16 [L][B][Hkv][nb_max][2][128], built from K
        by ``pool_all`` / the fill methods and kept current by ``append_tokens``)."""
        if scoring not in ("maxdot", "pooled"):
            raise ValueError(f"unknown scoring {scoring!r}")
        self.scoring = scoring
        self.w = w
        self.device = torch.device(device)
        self.L_phys = l_phys or w.L
        self.L_host = l_host or self.L_phys
        self.shape = B.Shape.from_workload(w)
        s = self.shape
        dev = self.device
        Lp = self.L_phys
        self.K = torch.zeros((Lp, s.B, s.Hkv, s.nb_max * 16, 128), dtype=torch.bfloat16, device=dev)
        self.Kp = (torch.zeros((Lp, s.B, s.Hkv, s.nb_max, 2, 128), dtype=torch.bfloat16, device=dev)
                   if scoring == "pooled" else None)
        self.k_pool = torch.zeros((Lp, s.B, s.Hkv, s.P, 16, 128), dtype=torch.bfloat16, device=dev)
        self.v_pool = torch.zeros_like(self.k_pool)
        self.blk2slot = torch.full((Lp, s.B, s.Hkv, s.nb_max), -1, dtype=torch.int32, device=dev)
        self.slot2blk = torch.full((Lp, s.B, s.Hkv, s.P), -1, dtype=torch.int32, device=dev)
        self.last_used = torch.full((Lp, s.B, s.Hkv, s.P), -1, dtype=torch.int32, device=dev)
        if host_alloc not in ("thp", "cuda", "thp_layers", "cuda_layers"):
            raise ValueError(f"unknown host_alloc {host_alloc!r}")
        self.pin_host, self.host_alloc = pin_host, host_alloc
        self._alloc_host()
        self.ctx = torch.tensor(w.ctx, dtype=torch.int32, device=dev)
        self.scratch = LayerScratch(s, dev)
        self.scratch2 = None
        self.step_dev = torch.zeros(1, dtype=torch.int32, device=dev)  # LRU clock read by the gather
        self.scale = 1.0 / math.sqrt(w.d)
        # per-layer views made once (indexing a tensor costs host time on every call)
        self.Kl = [self.K[l] for l in range(Lp)]
        self.Kpl = [self.Kp[l] for l in range(Lp)] if self.Kp is not None else None
        self.kpl = [self.k_pool[l] for l in range(Lp)]
        self.vpl = [self.v_pool[l] for l in range(Lp)]
        self.b2sl = [self.blk2slot[l] for l in range(Lp)]
        self.s2bl = [self.slot2blk[l] for l in range(Lp)]
        self.lul = [self.last_used[l] for l in range(Lp)]
        self.fused_select = True  # a2 + a3 in one launch (oasis_topk_select_diff) on the decode path
        # prefetching the fetched blocks' host data into L2 from that launch moved the
        # host-link latency into it (top-K + diff +15 us, gather -15 us): off
        self.prefetch_host = False
        # max-dot scoring through oasis_score_blocks_dynamic (chunks from an atomic
        # counter) instead of the fixed-stride persistent grid
        # max-dot scoring through oasis_score_blocks_dynamic (the mma.sync kernel with a
        # share of fixed ranges and chunks from an atomic counter) instead of the
        # default scorer; a pooled or copy-carrying launch ignores it
        self.dynamic_scorer = False
        self._lag_sel = None  # per-layer selections of the cross-step pipeline (copy="lag")
        self._lag_nsel = None
        self._lag_ready = False

    def _alloc_host(self):
        """The host tier, bf16 [L_host][B][Hkv][nb_max][2][16][128], page-locked and mapped."""
        s = self.shape
        host_shape = (self.L_host, s.B, s.Hkv, s.nb_max, 2, 16, 128)
        self._host_buf, self._host_bufs = None, None
        if self.pin_host and self.host_alloc == "thp":
            nbytes = int(np.prod(host_shape)) * 2
            self._host_buf = HugePinnedBuffer(nbytes)
            self.host = self._host_buf.tensor.view(torch.bfloat16).view(host_shape)
        elif self.pin_host and self.host_alloc == "cuda":  # page-locked by the CUDA allocator (cudaHostAlloc)
            self.host = torch.empty(host_shape, dtype=torch.bfloat16, pin_memory=True)
        elif self.pin_host:  # one allocation (and registration) per layer: "thp_layers" or "cuda_layers"
            per = host_shape[1:]
            if self.host_alloc == "thp_layers":
                self._host_bufs = [HugePinnedBuffer(int(np.prod(per)) * 2) for _ in range(self.L_host)]
                self.host = [b_.tensor.view(torch.bfloat16).view(per) for b_ in self._host_bufs]
            else:
                self.host = [torch.empty(per, dtype=torch.bfloat16, pin_memory=True) for _ in range(self.L_host)]
        else:
            self.host = torch.zeros(host_shape, dtype=torch.bfloat16)
        self.hostl = [self.host[l] for l in range(self.L_host)]

    def _free_host(self):
        self.hostl = None
        self.host = None
        for buf in ([self._host_buf] if self._host_buf is not None else []) + list(self._host_bufs or []):
            buf.close()
        self._host_buf, self._host_bufs = None, None

    def rebuild_host_tier(self, l_host: int):
        """Replace the host tier by one holding l_host layers (layer l then reads host
        buffer l mod l_host) and refill it from the generator.  Tables and HBM slots
        are left as they are (for timing: a slot keeps the data of the host buffer
        it was fetched from)."""
        torch.cuda.synchronize(self.device)
        self._free_host()
        empty = getattr(torch._C, "_host_emptyCache", None)  # return cached page-locked memory
        if empty is not None:
            empty()
        self.L_host = max(1, min(int(l_host), self.L_phys))
        self._alloc_host()
        w = self.w
        for layer in range(self.L_host):
            for b in range(w.B):
                Kr, Vr = syn.kv_request_torch(w, layer, b, self.device)
                kb = Kr.view(w.Hkv, w.nb_max, 16, 128)
                vb = Vr.view(w.Hkv, w.nb_max, 16, 128)
                self.hostl[layer][b].copy_(torch.stack([kb, vb], dim=2))
        torch.cuda.synchronize(self.device)

    # ---------------------------------------------------------------- filling
    def fill_layer_numpy(self, layer: int, K_bits: np.ndarray, V_bits: np.ndarray,
                         blk2slot: np.ndarray, slot2blk: np.ndarray, last_used: np.ndarray):
        """Load one layer from host arrays (bf16 bits [B][Hkv][T_max][d] and int32 tables)."""
        lp, lh = layer % self.L_phys, layer % self.L_host
        w = self.w
        self.K[lp].copy_(_bf16_from_bits(K_bits, self.device))
        host = syn.host_tier_from_kv(w, K_bits, V_bits)
        self.host[lh].copy_(torch.from_numpy(host.view(np.int16)).view(torch.bfloat16))
        self.blk2slot[lp].copy_(torch.from_numpy(blk2slot))
        self.slot2blk[lp].copy_(torch.from_numpy(slot2blk))
        self.last_used[lp].copy_(torch.from_numpy(last_used))
        kp, vp = syn.pools_from_tables(w, host, slot2blk)
        self.k_pool[lp].copy_(_bf16_from_bits(kp, self.device))
        self.v_pool[lp].copy_(_bf16_from_bits(vp, self.device))
        self.pool_layer(lp)

    def fill_synthetic(self):
        """Generate every layer on the device (keys, host tier, pools, tables).

        Uses the counter-based generator (bit-identical to the host one).  With
        a host tier of fewer layers than the model, only layers < L_host write
        the host tier; layer l's gathers read host buffer l mod L_host.
        """
        w = self.w
        dev = self.device
        ar = torch.arange(w.Hkv, device=dev)[:, None]
        for layer in range(w.L):
            lp, lh = layer % self.L_phys, layer % self.L_host
            b2s, s2b, lu = syn.initial_tables(w, layer)
            for b in range(w.B):
                Kr, Vr = syn.kv_request_torch(w, layer, b, dev)
                self.K[lp, b].copy_(Kr)
                kb = Kr.view(w.Hkv, w.nb_max, 16, 128)
                vb = Vr.view(w.Hkv, w.nb_max, 16, 128)
                if layer < self.L_host:
                    self.hostl[lh][b].copy_(torch.stack([kb, vb], dim=2))
                idx = torch.from_numpy(s2b[b]).to(dev).long()
                occ = (idx >= 0)[..., None, None]
                self.k_pool[lp, b].copy_(kb[ar, idx.clamp(min=0)] * occ)
                self.v_pool[lp, b].copy_(vb[ar, idx.clamp(min=0)] * occ)
            self.blk2slot[lp].copy_(torch.from_numpy(b2s))
            self.slot2blk[lp].copy_(torch.from_numpy(s2b))
            self.last_used[lp].copy_(torch.from_numpy(lu))
            self.pool_layer(lp)
        torch.cuda.synchronize(dev)

    def warm_host_tier(self, stream=None):
        """Read the whole host tier once through the SMs' zero-copy loads
        (oasis_touch_host), so that later gathers do not meet first-read stalls."""
        st = stream or torch.cuda.current_stream(self.device)
        for l in range(self.L_host):
            B.oasis_touch_host(self.hostl[l], stream=st)
        torch.cuda.synchronize(self.device)

    def set_scoring(self, scoring: str):
        """Switch the decode path between max-dot and pooled scoring.  The pooled key
        cache is made (and built from the current keys) on first use and then kept
        current by appends in either mode."""
        if scoring not in ("maxdot", "pooled"):
            raise ValueError(f"unknown scoring {scoring!r}")
        if scoring == "pooled" and self.Kp is None:
            s = self.shape
            self.Kp = torch.zeros((self.L_phys, s.B, s.Hkv, s.nb_max, 2, 128), dtype=torch.bfloat16,
                                  device=self.device)
            self.Kpl = [self.Kp[l] for l in range(self.L_phys)]
            for lp in range(self.L_phys):
                self.pool_layer(lp)
        self.scoring = scoring

    def pool_layer(self, lp: int, stream=None):
        """Rebuild layer lp's pooled keys from its full keys (pooled scoring only)."""
        if self.Kp is None:
            return
        B.oasis_pool_keys(self.shape, self.K[lp], self.ctx, self.Kp[lp],
                          stream or torch.cuda.current_stream(self.device))

    def fill_layer_synthetic(self, layer: int):
        """Generate one layer on the device with the counter-based generator."""
        lp, lh = layer % self.L_phys, layer % self.L_host
        w = self.w
        for b in range(w.B):
            for h in range(w.Hkv):
                Kh, Vh = syn.head_kv_torch(w, layer, b, h, self.device)
                self.K[lp, b, h].copy_(Kh)
                kv = torch.stack([Kh.view(w.nb_max, 16, 128), Vh.view(w.nb_max, 16, 128)], dim=1)
                self.hostl[lh][b, h].copy_(kv, non_blocking=False)
        b2s, s2b, lu = syn.initial_tables(w, layer)
        self.blk2slot[lp].copy_(torch.from_numpy(b2s))
        self.slot2blk[lp].copy_(torch.from_numpy(s2b))
        self.last_used[lp].copy_(torch.from_numpy(lu))
        # pools hold the initial residents
        s2b_t = torch.from_numpy(s2b).to(self.device).long()
        Kv = self.K[lp].view(w.B, w.Hkv, w.nb_max, 16, 128)
        idx = s2b_t.clamp(min=0)
        gathered = torch.gather(Kv, 2, idx[..., None, None].expand(-1, -1, -1, 16, 128))
        self.k_pool[lp].copy_(gathered * (s2b_t >= 0)[..., None, None])
        hostv = self.host[lh][:, :, :, 1].to(self.device)
        gv = torch.gather(hostv, 2, idx[..., None, None].expand(-1, -1, -1, 16, 128))
        self.v_pool[lp].copy_(gv * (s2b_t >= 0)[..., None, None])
        self.pool_layer(lp)

    # ---------------------------------------------------------------- one layer-step
    def layer_step(self, layer: int, q_la: torch.Tensor, q: torch.Tensor, step: int,
                   stream=None, gather_stream=None, scratch: Optional[LayerScratch] = None,
                   gather: str = "fused"):
        """Run a1..a5 for one layer: score, top-K, capped diff, gather, attention.

        q_la: bf16 [B][n_la][Hq][d], q: bf16 [B][Hq][d] (device).  Returns the
        scratch holding the outputs.  With ``gather_stream`` the gather runs on
        that stream and the attention waits for it.  ``gather`` picks how a4 is
        issued: "fused" (oasis_gather_h2d), "split" (oasis_assign_slots then
        oasis_copy_fetched) or "carry" (oasis_assign_slots, then the copy carried
        by a second scoring launch of the same layer, oasis_score_blocks_copy).
        """
        s = self.shape
        sc = scratch or self.scratch
        lp, lh = layer % self.L_phys, layer % self.L_host
        st = stream or torch.cuda.current_stream(self.device)
        step = self._step_tensor(step, st)
        K = self.K[lp]
        self._score_topk_diff(lp, q_la, sc, st, layer)
        gs = gather_stream or st
        if gs is not st:
            gs.wait_stream(st)
        if gather == "fused":
            B.oasis_gather_h2d(s, self.host[lh], sc.sel, sc.nsel, sc.fetch, sc.nfetch, self.blk2slot[lp],
                               self.slot2blk[lp], self.last_used[lp], step, self.k_pool[lp],
                               self.v_pool[lp], sc.err, gs)
        elif gather in ("split", "carry"):
            B.oasis_assign_slots(s, sc.sel, sc.nsel, sc.fetch, sc.nfetch, self.blk2slot[lp],
                                 self.slot2blk[lp], self.last_used[lp], step, sc.err, gs)
            if gather == "split":
                B.oasis_copy_fetched(s, self.host[lh], sc.fetch, sc.nfetch, self.blk2slot[lp],
                                     self.k_pool[lp], self.v_pool[lp], sc.err, gs)
            elif self.scoring == "pooled":
                B.oasis_score_blocks_pooled(s, self.Kp[lp], self.ctx, q_la, sc.scores, self.host[lh], sc.fetch,
                                            sc.nfetch, self.blk2slot[lp], self.k_pool[lp], self.v_pool[lp],
                                            sc.err, gs)
            else:
                B.oasis_score_blocks_copy(s, K, self.ctx, q_la, sc.scores, self.host[lh], sc.fetch,
                                          sc.nfetch, self.blk2slot[lp], self.k_pool[lp], self.v_pool[lp],
                                          sc.err, gs)
        else:
            raise ValueError(f"unknown gather mode {gather!r}")
        if gs is not st:
            st.wait_stream(gs)
        B.oasis_sparse_decode_attn(s, q, self.k_pool[lp], self.v_pool[lp], sc.sel, sc.nsel,
                                   self.blk2slot[lp], self.ctx, self.scale, sc.ws, sc.ws_bytes,
                                   sc.out, st)
        return sc

    # ---------------------------------------------------------------- one decode step
    def _step_tensor(self, step, stream):
        """The LRU clock as a device int32 scalar (an int is written into step_dev on `stream`)."""
        if isinstance(step, torch.Tensor):
            return step
        with torch.cuda.stream(stream):
            self.step_dev.fill_(int(step))
        return self.step_dev

    def _score_topk_diff(self, lp, q_la, sc, st, layer=None):
        self._select_lp(lp, q_la, sc, st, host_layer=layer)

    def _select(self, layer, q_la, step, sc, st, mark=None, carry=None):
        """a1..a3 of one layer; ``carry=(layer', scratch')`` makes the scoring launch
        also copy the fetched blocks of layer' (whose slots are already assigned)."""
        self._select_lp(layer % self.L_phys, q_la, sc, st, mark, carry, host_layer=layer)

    def _select_lp(self, lp, q_la, sc, st, mark=None, carry=None, host_layer=None):
        self._score_lp(lp, q_la, sc, st, mark, carry)
        self._topk_diff_lp(lp, q_la, sc, st, mark, host_layer)

    def _score_lp(self, lp, q_la, sc, st, mark=None, carry=None):
        s = self.shape
        pooled = self.scoring == "pooled"
        K = self.Kpl[lp] if pooled else self.Kl[lp]
        if mark:
            mark("score", st)
        if self.dynamic_scorer and not pooled and carry is None:
            B.oasis_score_blocks_dynamic(s, K, self.ctx, q_la, sc.scores, sc.work, 0, st)
        elif carry is None:
            if pooled:
                B.oasis_score_blocks_pooled(s, K, self.ctx, q_la, sc.scores, err_word=sc.err, stream=st)
            else:
                B.oasis_score_blocks(s, K, self.ctx, q_la, sc.scores, sc.err, st)
        else:
            cl, csc = carry
            clp, clh = cl % self.L_phys, cl % self.L_host
            args = (self.hostl[clh], csc.fetch, csc.nfetch, self.b2sl[clp], self.kpl[clp], self.vpl[clp], sc.err, st)
            if pooled:
                B.oasis_score_blocks_pooled(s, K, self.ctx, q_la, sc.scores, *args)
            else:
                B.oasis_score_blocks_copy(s, K, self.ctx, q_la, sc.scores, *args)

    def _topk_diff_lp(self, lp, q_la, sc, st, mark=None, host_layer=None):
        s = self.shape
        pooled = self.scoring == "pooled"
        K = self.Kpl[lp] if pooled else self.Kl[lp]
        if mark:
            mark("topk", st)
        if self.fused_select:
            f = B.oasis_topk_select_diff_pooled if pooled else B.oasis_topk_select_diff
            hl = lp if host_layer is None else host_layer
            hp = self.hostl[hl % self.L_host] if self.prefetch_host else None
            f(s, sc.scores, K, q_la, self.ctx, self.b2sl[lp], self.w.C, sc.sel, sc.nsel, sc.fetch, sc.nfetch, hp, st)
        else:
            topk = B.oasis_topk_select_pooled if pooled else B.oasis_topk_select
            diff = B.oasis_fetch_diff_capped_pooled if pooled else B.oasis_fetch_diff_capped
            topk(s, sc.scores, K, q_la, self.ctx, sc.sel, sc.nsel, st)
            if mark:
                mark("diff", st)
            diff(s, sc.scores, K, q_la, self.ctx, sc.sel, sc.nsel, self.b2sl[lp], self.w.C, sc.fetch, sc.nfetch,
                 st)
        if mark:
            mark("end", st)

    def _gather(self, layer, step, sc, gs):
        s = self.shape
        lp, lh = layer % self.L_phys, layer % self.L_host
        B.oasis_gather_h2d(s, self.hostl[lh], sc.sel, sc.nsel, sc.fetch, sc.nfetch, self.b2sl[lp],
                           self.s2bl[lp], self.lul[lp], step, self.kpl[lp], self.vpl[lp], sc.err, gs)

    def _assign(self, layer, step, sc, st):
        s = self.shape
        lp = layer % self.L_phys
        B.oasis_assign_slots(s, sc.sel, sc.nsel, sc.fetch, sc.nfetch, self.b2sl[lp], self.s2bl[lp],
                             self.lul[lp], step, sc.err, st)

    def _copy(self, layer, sc, st):
        """The data half of layer `layer`'s gather (its slots already assigned)."""
        s = self.shape
        lp, lh = layer % self.L_phys, layer % self.L_host
        B.oasis_copy_fetched(s, self.hostl[lh], sc.fetch, sc.nfetch, self.b2sl[lp], self.kpl[lp],
                             self.vpl[lp], sc.err, st)

    def _attend(self, layer, q, sc, st, out=None):
        s = self.shape
        lp = layer % self.L_phys
        B.oasis_sparse_decode_attn(s, q, self.kpl[lp], self.vpl[lp], sc.sel, sc.nsel, self.b2sl[lp],
                                   self.ctx, self.scale, sc.ws, sc.ws_bytes,
                                   sc.out if out is None else out, st)

    def attend_lookahead(self, layer: int, q: torch.Tensor, q_la: torch.Tensor, sc, out: torch.Tensor,
                         out_la: torch.Tensor, stream=None):
        """f2: the true and the lookahead queries of one layer over the resident
        blocks of sc's selection, in one launch (out [B][Hq][d], out_la
        [B][n_la][Hq][d], fp32)."""
        s = self.shape
        lp = layer % self.L_phys
        nbytes = B.oasis_attn_lookahead_workspace_bytes(s)
        if getattr(self, "_la_ws", None) is None or self._la_ws.numel() < nbytes:
            self._la_ws = torch.empty(max(16, nbytes), dtype=torch.uint8, device=self.device)
        B.oasis_sparse_decode_attn_lookahead(s, q, q_la, self.kpl[lp], self.vpl[lp], sc.sel, sc.nsel, self.b2sl[lp],
                                             self.ctx, self.scale, self._la_ws, nbytes, out, out_la,
                                             stream or torch.cuda.current_stream(self.device))

    def _tally(self, layer, sc, count, fetched):
        if count is not None:
            count.add_(self.attended_blocks(layer, sc))
        if fetched is not None:
            fetched.add_(sc.nfetch.sum())

    def attended_blocks(self, layer: int, sc: "LayerScratch") -> torch.Tensor:
        """Device count of attended blocks (selected and resident) of one layer, all heads."""
        lp = layer % self.L_phys
        sel = sc.sel.long()
        valid = (sel >= 0) & (torch.arange(self.shape.Kb, device=self.device) < sc.nsel[..., None])
        slot = torch.gather(self.b2sl[lp].long(), 2, sel.clamp(min=0))
        return ((slot >= 0) & valid).sum()

    def decode_step(self, step, q_la_layers, q_layers, out_layers=None, main=None, side=None,
                    mark=None, count=None, copy: str = "overlap", fetched=None):
        """All layers of one decode step, pipelined across layers.

        copy="overlap" (default): select(l) on ``main``, then the whole gather of
          layer l on a side stream while ``main`` runs attn(l-1); select(l+1)
          waits for gather(l).  The fastest order measured with a host tier from
          cudaHostAlloc.
        copy="carry", all on the main stream:
            score(0) topk(0) diff(0) assign(0)
            score(1)+copy(0) topk(1) diff(1) assign(1) attn(0)
            score(2)+copy(1) ...                         attn(1)
            ...  copy(L-1) attn(L-1)
          The table half of layer l's gather runs right after its selection; the
          host-link copy of layer l rides in layer l+1's scoring launch, whose
          HBM-bound work hides the link latency; attn(l) follows that launch.
        copy="pipe": the scorers of all layers back to back on ``main``; layer l's
          top-K + diff, gather and attention on a side stream once its scores
          exist, running beside the following scorers (a ring of 4 scratch sets).
        copy="lag": the cross-step pipeline (f4): attn(l) over the selection the
          previous step made for layer l, then select(l) and gather(l) for the next
          step; one stream.
        copy="fork": score(l) and top-K + diff(l) on ``main``; attn(l-1) on a side
          stream once score(l) is done (beside top-K(l)); gather(l) on a second side
          stream once top-K(l) is done; score(l+1) waits for both.
        copy="gather": select(0); select(1); attn(0); select(2); attn(1); ... with
          the whole gather (oasis_gather_h2d) of layer l right after select(l), on
          ``side`` if given (attn(l) then waits for it).
        Two scratch sets alternate between consecutive layers.  q_la_layers[l],
        q_layers[l]: device tensors of layer l; out_layers[l] (optional) receives
        the fp32 attention output of layer l.  ``mark(name, stream)``, if given, is
        called before each kernel ("score", "topk", "diff", "assign", "copy",
        "gather", "attn") and after the last one of a group ("end", "gather_end",
        "attn_end") so the caller can record CUDA events.
        """
        L = self.w.L
        main = main or torch.cuda.current_stream(self.device)
        step = self._step_tensor(step, main)
        if self.scratch2 is None:
            self.scratch2 = LayerScratch(self.shape, self.device)
        scr = (self.scratch, self.scratch2)

        def attend_on(l, stream_):
            if mark:
                mark("attn", stream_)
            self._attend(l, q_layers[l], scr[l % 2], stream_, None if out_layers is None else out_layers[l])
            if mark:
                mark("attn_end", stream_)
            if count is not None or fetched is not None:
                self._tally(l, scr[l % 2], count, fetched)

        def attend(l):
            if mark:
                mark("attn", main)
            self._attend(l, q_layers[l], scr[l % 2], main, None if out_layers is None else out_layers[l])
            if mark:
                mark("attn_end", main)
            if count is not None or fetched is not None:
                self._tally(l, scr[l % 2], count, fetched)

        if copy == "pipe":
            # scorers back to back on `main`; each layer's selection, gather and
            # attention on a side stream as soon as its scores exist, beside the
            # next scorers (which should leave SM room: OPT_SCORE_CTAS_PER_SM).
            # A ring of scratch sets; scorer l waits until layer l - R is done.
            side = side if (side is not None and side is not main) else self._side_stream()
            R = 4
            ring = self._pipe_ring(R)
            ev_score = [torch.cuda.Event() for _ in range(L)]
            ev_done = [torch.cuda.Event() for _ in range(L)]
            for l in range(L):
                sc = ring[l % R]
                lp = l % self.L_phys
                if l >= R:
                    main.wait_event(ev_done[l - R])
                self._score_lp(lp, q_la_layers[l], sc, main, mark)
                ev_score[l].record(main)
                side.wait_event(ev_score[l])
                self._topk_diff_lp(lp, q_la_layers[l], sc, side, mark, host_layer=l)
                if mark:
                    mark("gather", side)
                self._gather(l, step, sc, side)
                if mark:
                    mark("gather_end", side)
                if mark:
                    mark("attn", side)
                self._attend(l, q_layers[l], sc, side, None if out_layers is None else out_layers[l])
                if mark:
                    mark("attn_end", side)
                if count is not None or fetched is not None:
                    self._tally(l, sc, count, fetched)
                ev_done[l].record(side)
            main.wait_stream(side)
            return
        if copy == "lag":
            # f4: attn(l) over the blocks the previous step's lookahead selected (held
            # in per-layer buffers), then this step's selection and gather of layer l,
            # which only prepare the next step.  The first lagged step has no earlier
            # selection: it selects and gathers first, then attends, like "gather".
            if self._lag_sel is None:
                s_ = self.shape
                self._lag_sel = torch.full((self.L_phys, s_.B, s_.Hkv, s_.Kb), -1, dtype=torch.int32,
                                           device=self.device)
                self._lag_nsel = torch.zeros((self.L_phys, s_.B, s_.Hkv), dtype=torch.int32, device=self.device)
                self._lag_ready = False
            first = not self._lag_ready
            for l in range(L):
                lp = l % self.L_phys
                view = _SelView(scr[l % 2], self._lag_sel[lp], self._lag_nsel[lp])
                if not first:
                    if mark:
                        mark("attn", main)
                    self._attend(l, q_layers[l], view, main, None if out_layers is None else out_layers[l])
                    if mark:
                        mark("attn_end", main)
                    if count is not None or fetched is not None:
                        self._tally(l, view, count, fetched)
                self._select(l, q_la_layers[l], step, view, main, mark)
                if mark:
                    mark("gather", main)
                self._gather(l, step, view, main)
                if mark:
                    mark("gather_end", main)
                if first:
                    if mark:
                        mark("attn", main)
                    self._attend(l, q_layers[l], view, main, None if out_layers is None else out_layers[l])
                    if mark:
                        mark("attn_end", main)
                    if count is not None or fetched is not None:
                        self._tally(l, view, count, fetched)
            self._lag_ready = True
            return
        if copy == "carry":
            for l in range(L):
                self._select(l, q_la_layers[l], step, scr[l % 2], main, mark,
                             carry=None if l == 0 else (l - 1, scr[(l - 1) % 2]))
                if mark:
                    mark("assign", main)
                self._assign(l, step, scr[l % 2], main)
                if l > 0:
                    attend(l - 1)
            if mark:
                mark("copy", main)
            self._copy(L - 1, scr[(L - 1) % 2], main)
            attend(L - 1)
            return
        if copy == "fork":
            # main: score(l) topk(l); side A: attn(l-1) once score(l) is done (beside
            # topk(l)); side B: gather(l) once topk(l) is done.  score(l+1) waits for
            # gather(l) and attn(l-1).
            sa = self._side_stream()
            sb = self._side_stream2()
            ev_sc = [torch.cuda.Event() for _ in range(2)]
            ev_sel = [torch.cuda.Event() for _ in range(2)]
            ev_gat = [torch.cuda.Event() for _ in range(2)]
            ev_att = [torch.cuda.Event() for _ in range(2)]
            for l in range(L):
                sc = scr[l % 2]
                lp = l % self.L_phys
                self._score_lp(lp, q_la_layers[l], sc, main, mark)
                if l > 0:
                    ev_sc[l % 2].record(main)
                    sa.wait_event(ev_sc[l % 2])
                    attend_on(l - 1, sa)
                    ev_att[l % 2].record(sa)
                self._topk_diff_lp(lp, q_la_layers[l], sc, main, mark, host_layer=l)
                ev_sel[l % 2].record(main)
                sb.wait_event(ev_sel[l % 2])
                if mark:
                    mark("gather", sb)
                self._gather(l, step, sc, sb)
                if mark:
                    mark("gather_end", sb)
                ev_gat[l % 2].record(sb)
                main.wait_event(ev_gat[l % 2])
                if l > 0:
                    main.wait_event(ev_att[l % 2])
            attend(L - 1)
            return
        if copy == "overlap":
            # main: S(l) [A(l-1)] wait G(l) S(l+1) ...; side: G(l) once S(l) is done.
            # G(l) overlaps A(l-1) only: the next scoring launch waits for it, so the
            # persistent scorer never shares the GPU with the gather.  A(l-1) is
            # issued before G(l): captured the other way round, the replayed graph
            # started A(l-1) only as G(l) ended (globaltimer spans of both kernels:
            # ~22 us after S(l) instead of ~2.5 us).
            side = side if (side is not None and side is not main) else self._side_stream()
            ev_sel = [torch.cuda.Event() for _ in range(2)]
            ev_gat = [torch.cuda.Event() for _ in range(2)]
            for l in range(L):
                sc = scr[l % 2]
                self._select(l, q_la_layers[l], step, sc, main, mark)
                ev_sel[l % 2].record(main)
                if l > 0:
                    attend(l - 1)
                side.wait_event(ev_sel[l % 2])
                if mark:
                    mark("gather", side)
                self._gather(l, step, sc, side)
                if mark:
                    mark("gather_end", side)
                ev_gat[l % 2].record(side)
                main.wait_event(ev_gat[l % 2])
            attend(L - 1)
            return
        if copy != "gather":
            raise ValueError(f"unknown copy mode {copy!r}")
        side = side or main
        events = [torch.cuda.Event() for _ in range(2)]

        def launch_select_gather(l):
            sc = scr[l % 2]
            self._select(l, q_la_layers[l], step, sc, main, mark)
            if side is not main:
                side.wait_stream(main)
            if mark:
                mark("gather", side)
            self._gather(l, step, sc, side)
            if mark:
                mark("gather_end", side)
            if side is not main:
                events[l % 2].record(side)

        launch_select_gather(0)
        for l in range(L):
            if l + 1 < L:
                launch_select_gather(l + 1)
            if side is not main:
                main.wait_event(events[l % 2])
            attend(l)

    def error_word(self) -> int:
        """OR of the device error words of every scratch set (synchronizes)."""
        sets = [self.scratch] + ([self.scratch2] if self.scratch2 is not None else []) + list(
            getattr(self, "_ring", None) or [])
        v = 0
        for sc in sets:
            v |= int(sc.err.item())
        return v

    def _pipe_ring(self, R: int):
        if getattr(self, "_ring", None) is None or len(self._ring) < R:
            self._ring = [self.scratch, self.scratch2] + [LayerScratch(self.shape, self.device) for _ in range(R - 2)]
        return self._ring[:R]

    def _side_stream2(self):
        if getattr(self, "_side2", None) is None:
            self._side2 = torch.cuda.Stream(self.device)
        return self._side2

    def _side_stream(self):
        if getattr(self, "_side", None) is None:
            self._side = torch.cuda.Stream(self.device)
        return self._side

    # ---------------------------------------------------------------- appends
    def append_step(self, k_new: torch.Tensor, v_new: torch.Tensor, stream=None):
        """One decode step's new token of every request in every layer (bf16
        [L][B][Hkv][d] each); ctx advances once, with the last layer."""
        L = self.w.L
        st = stream or torch.cuda.current_stream(self.device)
        if self.Kp is not None:  # every layer's token becomes valid when ctx advances below
            for l in range(L):
                B.oasis_pool_append(self.shape, k_new[l], self.ctx, self.Kp[l % self.L_phys], self.scratch.err, st)
        for l in range(L):
            lp, lh = l % self.L_phys, l % self.L_host
            B.oasis_append_kv(self.shape, k_new[l], v_new[l], self.ctx, self.K[lp], self.host[lh], self.blk2slot[lp],
                              self.k_pool[lp], self.v_pool[lp], l == L - 1, self.scratch.err, st)

    def append_tokens(self, layer: int, k_new: torch.Tensor, v_new: torch.Tensor, advance: bool,
                      stream=None, err=None):
        """Append one token per request (bf16 [B][Hkv][d]) to layer `layer`'s caches.

        With pooled scoring the token is folded into its block's pooled keys only
        when ``advance`` makes it valid; after advancing ctx some other way, call
        ``pool_layer``."""
        lp, lh = layer % self.L_phys, layer % self.L_host
        st = stream or torch.cuda.current_stream(self.device)
        if self.Kp is not None and advance:  # before the append advances ctx
            B.oasis_pool_append(self.shape, k_new, self.ctx, self.Kp[lp], self.scratch.err if err is None else err, st)
        B.oasis_append_kv(self.shape, k_new, v_new, self.ctx, self.K[lp], self.host[lh], self.blk2slot[lp],
                          self.k_pool[lp], self.v_pool[lp], advance,
                          self.scratch.err if err is None else err, st)


class AgreementProbe:
    """Per-layer agreement of predicted top-K sets with the exact one (f3).

    For one layer and step: the exact set E = top-K of the true queries (the
    max-dot block score with the true query as the only lookahead row), the
    lookahead prediction S_la = top-K of the lookahead queries, and optionally
    the previous-token prediction S_prev = top-K of the previous step's true
    queries (both predictions with the decode path's scoring, max-dot or pooled); oasis_set_agreement then counts |S & E| (and |S & E & resident|)
    per head.  Uses its own buffers; the decode state's tables are only read.
    """

    def __init__(self, st: "DecodeState", K: Optional[int] = None):
        s = st.shape
        self.st = st
        self.K = K or s.Kb
        self.shape = B.Shape(s.B, s.Hq, s.Hkv, s.d, s.bs, s.nb_max, s.n_la, self.K, max(s.P, self.K))
        self.shape1 = B.Shape(s.B, s.Hq, s.Hkv, s.d, s.bs, s.nb_max, 1, self.K, max(s.P, self.K))
        dev = st.device
        self.scores = torch.empty((s.B, s.Hkv, s.nb_max, 2), dtype=torch.float32, device=dev)
        self.sel = {k: torch.empty((s.B, s.Hkv, self.K), dtype=torch.int32, device=dev)
                    for k in ("exact", "la", "prev")}
        self.nsel = {k: torch.empty((s.B, s.Hkv), dtype=torch.int32, device=dev) for k in self.sel}
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)

    def _topk(self, shape, layer, q_rows, which, stream, pooled=False):
        st = self.st
        lp = layer % st.L_phys
        if pooled:
            Kp = st.Kpl[lp]
            B.oasis_score_blocks_pooled(shape, Kp, st.ctx, q_rows, self.scores, err_word=self.err, stream=stream)
            B.oasis_topk_select_pooled(shape, self.scores, Kp, q_rows, st.ctx, self.sel[which], self.nsel[which],
                                       stream)
            return
        K = st.Kl[lp]
        B.oasis_score_blocks(shape, K, st.ctx, q_rows, self.scores, self.err, stream)
        B.oasis_topk_select(shape, self.scores, K, q_rows, st.ctx, self.sel[which], self.nsel[which], stream)

    def run(self, layer: int, q_la: torch.Tensor, q: torch.Tensor, q_prev: Optional[torch.Tensor] = None,
            stream=None):
        """Counts [B][Hkv][3] for the lookahead prediction (and the previous-token one)."""
        st = self.st
        stream = stream or torch.cuda.current_stream(st.device)
        pooled = st.scoring == "pooled"  # the predictors score as the decode path does
        self._topk(self.shape1, layer, q, "exact", stream)
        self._topk(self.shape, layer, q_la, "la", stream, pooled)
        b2s = st.b2sl[layer % st.L_phys]
        out = {}
        for which, q_pred in (("la", None), ("prev", q_prev)):
            if which == "prev":
                if q_pred is None:
                    continue
                self._topk(self.shape1, layer, q_pred, "prev", stream, pooled)
            counts = torch.empty((self.shape.B, self.shape.Hkv, 3), dtype=torch.int32, device=st.device)
            B.oasis_set_agreement(self.shape, self.sel[which], self.nsel[which], self.sel["exact"],
                                  self.nsel["exact"], b2s, counts, self.err, stream)
            out[which] = counts
        return out


class KernelTrace:
    """Kernel span records (oasis_trace_set) in a device buffer owned here.

    ``start()`` makes later launches record (a CUDA graph captured meanwhile keeps
    recording on every replay), ``stop()`` ends that for new launches,
    ``spans()`` returns, per kind, the (start, end) nanosecond arrays of the
    recorded launches in launch order.  Diagnostics only: results do not depend on
    it.
    """

    KINDS = {"score": B.TRACE_SCORE, "score_pooled": B.TRACE_SCORE_POOLED, "select": B.TRACE_SELECT,
             "gather": B.TRACE_GATHER, "copy": B.TRACE_COPY, "attn": B.TRACE_ATTN, "append": B.TRACE_APPEND}

    def __init__(self, capacity: int = 1024, device="cuda"):
        self.capacity = int(capacity)
        nbytes = B.oasis_trace_bytes(self.capacity)
        self.buf = torch.zeros((nbytes + 7) // 8, dtype=torch.int64, device=device)

    def start(self):
        B.oasis_trace_set(self.buf, self.capacity)

    @staticmethod
    def stop():
        B.oasis_trace_set(None)

    def reset(self):
        self.buf.zero_()

    def spans(self):
        raw = self.buf.cpu().numpy().view(np.uint8)
        ctl = raw[:B.TRACE_HEADER_BYTES].view(np.uint32)[:2 * B.TRACE_KINDS]
        rec = raw[B.TRACE_HEADER_BYTES:B.TRACE_HEADER_BYTES + B.TRACE_KINDS * self.capacity * 16]
        rec = rec.view(np.uint64).reshape(B.TRACE_KINDS, self.capacity, 2)
        out = {}
        for name, k in self.KINDS.items():
            n = int(ctl[2 * k])
            if n > self.capacity:
                raise RuntimeError(f"{n} launches of kind {name} overflowed a trace of {self.capacity} records")
            out[name] = ((~rec[k, :n, 0]).astype(np.int64), rec[k, :n, 1].astype(np.int64))
        return out


class StepGraph:
    """Decode steps captured as one CUDA graph and replayed.

    ``q_la_steps[k]`` / ``q_steps[k]`` are the device inputs of captured step k
    (per-layer tensors or [L]-leading tensors) and ``out_steps[k]`` its [L]-leading
    fp32 output.  The LRU clock ``step`` (device int32 [1]) starts at
    ``first_step`` and the graph itself advances it after every step, so each
    replay continues the decode.  ``mark`` (as for decode_step) is called during
    capture; CUDA events recorded by it become nodes of the graph.
    """

    def __init__(self, st: DecodeState, first_step: int, q_la_steps, q_steps, out_steps, mark=None,
                 copy: str = "overlap", appends=None):
        self.st = st
        dev = st.device
        if st.scratch2 is None:
            st.scratch2 = LayerScratch(st.shape, dev)
        self.step = torch.full((1,), int(first_step), dtype=torch.int32, device=dev)
        self.graph = torch.cuda.CUDAGraph()
        self.stream = torch.cuda.Stream(dev)
        self.stream.wait_stream(torch.cuda.current_stream(dev))
        torch.cuda.synchronize(dev)
        with torch.cuda.graph(self.graph, stream=self.stream):
            for k in range(len(q_steps)):
                if appends is not None:  # (k_new, v_new) of captured step k: the growing context
                    st.append_step(appends[k][0], appends[k][1], stream=self.stream)
                st.decode_step(self.step, q_la_steps[k], q_steps[k], out_layers=out_steps[k],
                               main=self.stream, side=self.stream, mark=mark, copy=copy)
                self.step.add_(1)
        torch.cuda.synchronize(dev)

    def replay(self):
        self.graph.replay()
