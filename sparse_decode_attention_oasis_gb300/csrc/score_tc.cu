// a1 on the 5th-generation tensor cores: TMA -> shared memory -> tcgen05.mma -> TMEM.
//
// Same definition and certified bound as score.cu (OasisKV, metalmedia.ai page,
// Figure 7 caption: the draft queries are matched against the keys to choose the
// next step's top-K blocks).  Persistent, warp-specialised, two CTAs per SM (one
// CTA per SM, with a 4-stage ring, streamed only 84% of the measured copy peak:
// a single producer-MMA-epilogue pipeline per SM does not keep enough loads in
// flight; two pipelines of 2 stages reach it):
//   warp 0      TMA producer: per 128-token tile, two 64-column boxes of keys
//               (SWIZZLE_128B) and the head's N lookahead-query rows, into a
//               2-stage ring; completion counted on a "full" mbarrier;
//   warp 1      owns 64 TMEM columns; one lane issues 8 x tcgen05.mma
//               (M=128 tokens, N=16|32 queries, K=16, bf16 -> fp32) per tile into
//               one of two TMEM accumulators and commits to the stage's "empty"
//               and the accumulator's "tfull" mbarriers;
//   warps 2..9  epilogue, two groups of four: group g takes the tiles that
//               went to accumulator g, so two tiles' epilogues overlap; a warp
//               reads its 32 TMEM lanes (one token per thread) with tcgen05.ld,
//               takes the masked max over the valid queries and the token's key
//               norm from the swizzled shared-memory tile (four independent
//               partial sums), reduces over 16 lanes per block and stores
//               (score, bound).
// Every mbarrier wait is bounded: on expiry the CTA raises OASIS_EW_TIMEOUT in the
// error word, stops, waits (bounded) for its own TMA copies and MMAs, frees TMEM
// and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"

namespace oasis {
namespace tc {

constexpr int kStages = 2;  // per CTA; two CTAs per SM
constexpr int kEpiGroups = 2;
constexpr int kThreads = 64 + kEpiGroups * 128;
// one 32-column TMEM accumulator per epilogue group (an allocation is a power of two >= 32)
constexpr uint32_t kTmemCols = kEpiGroups <= 2 ? 64u : (kEpiGroups <= 4 ? 128u : 256u);
constexpr uint32_t kKBox = 128 * 128;                    // 128 rows x 128 B
constexpr uint32_t kQBox = 32 * 128;                     // up to 32 rows x 128 B
constexpr uint32_t kStageBytes = 2 * kKBox + 2 * kQBox;  // 40 KiB, multiple of 1024
constexpr unsigned long long kWaitNs = 2000000000ull;  // a wait gives up after 2 s

struct Bars {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t tfull[kEpiGroups];
  uint64_t tempty[kEpiGroups];
  uint32_t tmem_base;
  int abort_flag;
};

constexpr size_t kSmemBytes = 1024 + (size_t)kStages * kStageBytes + sizeof(Bars);

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* b, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(b)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* b) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(b)) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* b, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(b)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try(uint64_t* b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred P;\n mbarrier.try_wait.parity.shared::cta.b64 P, [%1], %2;\n selp.b32 %0, 1, 0, P;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(b)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// Bounded wait (kWaitNs of wall time); false when it expires or another role aborted.
__device__ __forceinline__ bool mbar_wait(uint64_t* b, uint32_t parity, volatile int* abort_flag) {
  if (mbar_try(b, parity)) return true;
  const unsigned long long t0 = global_ns();
  unsigned n = 0;
  while (!mbar_try(b, parity)) {
    if ((++n & 63u) == 0 && (*abort_flag || global_ns() - t0 > kWaitNs)) return false;
  }
  return true;
}

// Bounded wait that ignores the abort flag (used while draining).
__device__ __forceinline__ void mbar_drain(uint64_t* b, uint32_t parity) {
  const unsigned long long t0 = global_ns();
  unsigned n = 0;
  while (!mbar_try(b, parity)) {
    if ((++n & 63u) == 0 && global_ns() - t0 > kWaitNs) return;
  }
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int c0, int c1, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
      ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int c0, int c1, int c2,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
      "[%5];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
      : "memory");
}

// K-major operand in a 128-byte swizzled tile: 8-row atoms of 1024 B (SBO), LBO unused.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)1 << 16;
  d |= (uint64_t)(1024u >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// kind::f16, bf16 x bf16 -> fp32, both operands K-major, M = 128.
__host__ __device__ constexpr uint32_t instr_desc(int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n"
      ::"r"(tmem_d), "l"(a), "l"(b), "r"(idesc), "r"(acc));
}

__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float* v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ uint4 lds16(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}

// sum of squares of one 128-element bf16 row held as two swizzled 128-byte rows
__device__ __forceinline__ float row_sumsq(uint32_t box0, uint32_t box1, int row) {
  float ss[4] = {0.f, 0.f, 0.f, 0.f};  // independent chains: one per word of a 16-byte chunk
#pragma unroll
  for (int bx = 0; bx < 2; ++bx) {
    const uint32_t base = (bx ? box1 : box0) + row * 128;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const uint4 v = lds16(base + ((c ^ (row & 7)) << 4));
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        ss[m] = fmaf(bf_lo(w[m]), bf_lo(w[m]), ss[m]);
        ss[m] = fmaf(bf_hi(w[m]), bf_hi(w[m]), ss[m]);
      }
    }
  }
  return (ss[0] + ss[1]) + (ss[2] + ss[3]);
}

// The valid 128-token tiles of all heads, in (request, KV head, tile) order, form
// one sequence (an exclusive prefix over requests in shared memory, B <= 512;
// above that every head gets tiles_per_head positions and the ones past its
// context are skipped); CTA c takes the c-th of gridDim.x equal contiguous ranges.
constexpr int kTcMaxPrefix = 512;

struct TileSeq {
  const int* pre;  // shared, [B + 1] when exact
  int B, Hkv, tiles_per_head;
  bool exact;
  __device__ void locate(int idx, int& head, int& t) const {
    if (!exact) {
      head = idx / tiles_per_head;
      t = idx - head * tiles_per_head;
      return;
    }
    int lo = 0, hi = B - 1;  // the last b with pre[b] <= idx (that request has tiles)
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (pre[mid] <= idx) lo = mid; else hi = mid - 1;
    }
    const int tb = (pre[lo + 1] - pre[lo]) / Hkv;
    if (tb <= 0) {  // idx past the sequence (an empty range): nothing is read there
      head = lo * Hkv;
      t = 0;
      return;
    }
    const int local = idx - pre[lo];
    const int h = local / tb;
    head = lo * Hkv + h;
    t = local - h * tb;
  }
};

// Walks a CTA's range of the sequence one tile at a time: located once, then each
// step adds one (the single producer and MMA threads see no search or division
// per tile; the context length is read again only when the request changes).
struct TileIter {
  const TileSeq& seq;
  const int* ctx_len;
  int nb_max;
  int b, h, t, tb, ctx, nb;
  __device__ TileIter(const TileSeq& q, const int* cl, int nbm, int idx) : seq(q), ctx_len(cl), nb_max(nbm) {
    int head;
    seq.locate(idx, head, t);
    b = head / seq.Hkv;
    h = head - b * seq.Hkv;
    load();
  }
  __device__ void load() {
    ctx = ctx_len[b];
    nb = clamp_nb(ctx, nb_max);
    tb = seq.exact ? (seq.pre[b + 1] - seq.pre[b]) / seq.Hkv : seq.tiles_per_head;
  }
  __device__ void next() {
    if (++t < tb) return;
    t = 0;
    if (++h < seq.Hkv) return;
    h = 0;
    ++b;
    if (b < seq.B) load();
    while (seq.exact && b < seq.B && tb == 0) {  // requests without tiles own no positions
      ++b;
      if (b < seq.B) load();
    }
  }
  __device__ int head() const { return b * seq.Hkv + h; }
  __device__ bool valid() const { return t * 8 < nb; }
};

__global__ void __launch_bounds__(kThreads, 2)
score_blocks_tc_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_q,
                       Shape s, const int* __restrict__ ctx_len, float2* __restrict__ scores,
                       unsigned* __restrict__ err, int tiles_per_head, int total_tiles, int npad,
                       float inv_sqrt_d, TraceBuf tb) {
  TraceScope trace_(tb, OASIS_TRACE_SCORE);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Bars* bars = reinterpret_cast<Bars*>(smem + (size_t)kStages * kStageBytes);
  volatile int* abort_flag = &bars->abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = s.Hq / s.Hkv;
  const int N = s.n_la * G;
  __shared__ int tpre[kTcMaxPrefix + 1];
  __shared__ int wsum[kThreads / 32];
  const TileSeq seq{tpre, s.B, s.Hkv, tiles_per_head, s.B <= kTcMaxPrefix};
  int seq_total = total_tiles;
  if (seq.exact) {
    int run = 0;
    for (int b0 = 0; b0 < s.B; b0 += kThreads) {
      const int b = b0 + threadIdx.x;
      const int n = b < s.B ? (clamp_nb(ctx_len[b], s.nb_max) + 7) / 8 * s.Hkv : 0;
      int x = n;  // inclusive scan over the CTA
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      if (lane == 31) wsum[warp] = x;
      __syncthreads();
      int off = 0, tot = 0;
      for (int w = 0; w < kThreads / 32; ++w) {
        off += w < warp ? wsum[w] : 0;
        tot += wsum[w];
      }
      if (b < s.B) tpre[b] = run + off + x - n;
      run += tot;
      __syncthreads();  // wsum is rewritten by the next round
    }
    if (threadIdx.x == 0) tpre[s.B] = run;
    __syncthreads();
    seq_total = tpre[s.B];
  }
  const int t_start = (int)((long long)blockIdx.x * seq_total / gridDim.x);
  const int t_end = (int)((long long)(blockIdx.x + 1) * seq_total / gridDim.x);

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&bars->full[i], 1);
      mbar_init(&bars->empty[i], 5);
    }
    for (int i = 0; i < kEpiGroups; ++i) {
      mbar_init(&bars->tfull[i], 1);
      mbar_init(&bars->tempty[i], 4);
    }
    bars->abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 ::"r"(smem_u32(&bars->tmem_base)), "r"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  bool timed_out = false;
  int done_tiles = 0;  // tiles this role finished (valid ones)

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint32_t tx = 2 * kKBox + 2 * (uint32_t)N * 128;
      int i = 0;
      TileIter it(seq, ctx_len, s.nb_max, t_start);
      for (int idx = t_start; idx < t_end; ++idx, it.next()) {
        if (!it.valid()) continue;
        const int head = it.head(), b = it.b, h = it.h, t = it.t;
        const int st = i % kStages, r = i / kStages;
        if (!mbar_wait(&bars->empty[st], (r & 1) ^ 1, abort_flag)) { timed_out = true; break; }
        uint8_t* buf = smem + (size_t)st * kStageBytes;
        mbar_expect_tx(&bars->full[st], tx);
        const int row0 = (int)((long long)head * s.nb_max * kBS + (long long)t * 128);
        tma_load_2d(buf, &tmap_k, 0, row0, &bars->full[st]);
        tma_load_2d(buf + kKBox, &tmap_k, 64, row0, &bars->full[st]);
        tma_load_3d(buf + 2 * kKBox, &tmap_q, 0, h * G, b * s.n_la, &bars->full[st]);
        tma_load_3d(buf + 2 * kKBox + kQBox, &tmap_q, 64, h * G, b * s.n_la, &bars->full[st]);
        ++i;
      }
      done_tiles = i;
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = instr_desc(npad);
      int i = 0;
      TileIter it(seq, ctx_len, s.nb_max, t_start);
      for (int idx = t_start; idx < t_end; ++idx, it.next()) {
        if (!it.valid()) continue;
        const int st = i % kStages, r = i / kStages, a = i % kEpiGroups, u = i / kEpiGroups;
        if (!mbar_wait(&bars->tempty[a], (u & 1) ^ 1, abort_flag)) { timed_out = true; break; }
        if (!mbar_wait(&bars->full[st], r & 1, abort_flag)) { timed_out = true; break; }
        tc_fence_after();
        const uint32_t kb = smem_u32(smem + (size_t)st * kStageBytes);
        const uint32_t qb = kb + 2 * kKBox;
        const uint32_t d = tmem + (uint32_t)(a * 32);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t off = (uint32_t)(kk & 3) * 32u;
          const uint64_t ad = smem_desc(kb + (uint32_t)(kk >> 2) * kKBox + off);
          const uint64_t bd = smem_desc(qb + (uint32_t)(kk >> 2) * kQBox + off);
          mma_bf16(d, ad, bd, idesc, kk > 0 ? 1u : 0u);
        }
        mma_commit(&bars->empty[st]);
        mma_commit(&bars->tfull[a]);
        ++i;
      }
      done_tiles = i;
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int quarter = warp & 3;  // the TMEM lanes this warp may read
    const int group = (warp - 2) >> 2;
    const int row = quarter * 32 + lane;
    int i = 0;
    int cached_head = -1;
    float qnorm = 0.f;
    TileIter it(seq, ctx_len, s.nb_max, t_start);
    for (int idx = t_start; idx < t_end; ++idx, it.next()) {
      if (!it.valid()) continue;
      const int head = it.head(), t = it.t, ctx = it.ctx, nb = it.nb;
      const int st = i % kStages, r = i / kStages, a = i % kEpiGroups, u = i / kEpiGroups;
      if (a != group) {  // the other group's tile
        ++i;
        continue;
      }
      bool ok = mbar_wait(&bars->tfull[a], u & 1, abort_flag);
      ok = ok && mbar_wait(&bars->full[st], r & 1, abort_flag);
      if (!__all_sync(0xffffffffu, ok)) { timed_out = true; break; }
      tc_fence_after();
      float acc[32];
      const uint32_t taddr = tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(a * 32);
      tmem_ld16(taddr, acc);
      if (npad > 16) tmem_ld16(taddr + 16, acc + 16);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->tempty[a]);
      const uint32_t kb = smem_u32(smem + (size_t)st * kStageBytes);
      const uint32_t qb = kb + 2 * kKBox;
      float kss = row_sumsq(kb, kb + kKBox, row);
      if (head != cached_head) {
        float qss = lane < N ? row_sumsq(qb, qb + kQBox, lane) : 0.f;
        qnorm = sqrtf(warp_max(qss));
        cached_head = head;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->empty[st]);
      const int tok = t * 128 + row;
      const bool valid = tok < ctx;
      float m = neg_inf();
#pragma unroll
      for (int n = 0; n < 32; ++n)
        if (n < N && valid) m = fmaxf(m, acc[n]);
      float kn2 = valid ? kss : 0.f;
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) {
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        kn2 = fmaxf(kn2, __shfl_xor_sync(0xffffffffu, kn2, o));
      }
      const int blk = (t * 128 + quarter * 32 + (lane & 16)) / kBS;
      if ((lane & 15) == 0 && blk < nb) {
        const float sc = m * inv_sqrt_d;
        const float e = kAccRel * 1.0009765625f * qnorm * sqrtf(kn2) * inv_sqrt_d +
                        fabsf(sc) * 2.384185791015625e-07f + 8.673617379884035e-19f;
        scores[(long long)head * s.nb_max + blk] = make_float2(sc, e);
      }
      ++i;
    }
    done_tiles = i;
  }

  if (timed_out) {
    *abort_flag = 1;
    if (lane == 0 && err) atomicOr(err, OASIS_EW_TIMEOUT);
  }
  // drain: the producer waits for the copies it issued, the MMA lane for its last commit
  if (warp == 0 && lane == 0) {
    for (int j = max(0, done_tiles - kStages); j < done_tiles; ++j)
      mbar_drain(&bars->full[j % kStages], (j / kStages) & 1);
  }
  if (warp == 1 && lane == 0 && done_tiles > 0) {
    const int j = done_tiles - 1;
    mbar_drain(&bars->tfull[j % kEpiGroups], (j / kEpiGroups) & 1);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
  }
}

// ------------------------------------------------------------------ host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

}  // namespace tc

// The key tensor map addresses rows with 32-bit coordinates.
bool score_tc_fits(const Shape& s) { return (long long)s.B * s.Hkv * s.nb_max * kBS <= 0x7fffffffLL; }

cudaError_t launch_score_blocks_tc(const Shape& s, const uint16_t* k, const int* ctx, const uint16_t* q_la,
                                   float2* scores, unsigned* err, cudaStream_t stream) {
  using namespace tc;
  auto enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  const int G = s.Hq / s.Hkv;
  const int N = s.n_la * G;
  const int npad = N <= 16 ? 16 : 32;
  CUtensorMap mk, mq;
  {
    const cuuint64_t dims[2] = {(cuuint64_t)kD, (cuuint64_t)s.B * s.Hkv * s.nb_max * kBS};
    const cuuint64_t strides[1] = {(cuuint64_t)kD * 2};
    const cuuint32_t box[2] = {64, 128};
    const cuuint32_t es[2] = {1, 1};
    if (enc(&mk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(k), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  {
    const cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)s.Hq, (cuuint64_t)s.B * s.n_la};
    const cuuint64_t strides[2] = {(cuuint64_t)kD * 2, (cuuint64_t)s.Hq * kD * 2};
    const cuuint32_t box[3] = {64, (cuuint32_t)G, (cuuint32_t)s.n_la};
    const cuuint32_t es[3] = {1, 1, 1};
    if (enc(&mq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<uint16_t*>(q_la), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  const int tiles_per_head = (s.nb_max + 7) / 8;
  const int total = s.B * s.Hkv * tiles_per_head;
  const int sms = sm_count();
  const int grid = total < 2 * sms ? total : 2 * sms;  // two CTAs per SM
  static int attr_cache[kMaxDevicesCached] = {};
  cudaError_t e = ensure_dyn_smem((const void*)score_blocks_tc_kernel, kSmemBytes, attr_cache);
  if (e != cudaSuccess) return e;
  score_blocks_tc_kernel<<<grid, kThreads, kSmemBytes, stream>>>(mk, mq, s, ctx, scores, err, tiles_per_head,
                                                                 total, npad, 1.0f / sqrtf((float)s.d),
                                                                 trace_buf());
  return cudaGetLastError();
}

}  // namespace oasis
