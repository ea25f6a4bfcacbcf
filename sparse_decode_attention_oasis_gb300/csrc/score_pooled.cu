// f1: block scoring from the min/max pooled keys, on the tensor cores.
//
// metalmedia.ai page, Figure 7 caption: the draft query scans the compressed
// (per-block min/max pooled) keys to predict the next step's top-K blocks.
// With hi/lo the pooled rows of block x, the pooled score of query n is the
// largest q.k any key inside the box [lo, hi] can reach:
//   P_n(x) = sum_i max(q_i hi_i, q_i lo_i) = sum_i q+_i hi_i + sum_i q-_i lo_i,
// q+ = max(q, 0), q- = min(q, 0) (lo <= hi).  So P_n(x) = q'.k' with
// q' = [q+ | q-] and k' = [hi | lo], a 256-long dot product, and a block is ONE
// 256-element row: one warp scores a tile of 16 blocks as a 16 x N tile
// D = K' (16 x 256) * Q'^T (256 x N) with mma.m16n8k16 (bf16 in, fp32 accumulate).
// score(x) = max over lookahead j and group heads g of P / sqrt(d).  The reads are
// 512 bytes per block instead of 4 KiB.
//
// Streaming.  A tile (16 consecutive blocks of one head) is 8 KiB of contiguous
// memory; each thread loads its A fragments of a tile straight into registers
// with sixteen 16-byte loads (every warp instruction covers full 32-byte
// sectors), 4 CTAs of 4 warps per SM, and reloads each chunk's registers with
// the same chunk of its next tile as soon as the chunk's MMAs are issued.  (A cp.async shared-memory ring per warp
// reached only 4.3 TB/s with no MMA at all: the register loads stream faster.)
//
// Work split.  The valid tiles of all heads (ceil(nb_b / 16) per head of request
// b) form one sequence in (request, KV head, tile) order; CTA c takes an equal
// contiguous share and its warps interleave over it, so heads with short
// contexts cost nothing and every CTA gets the same number of tiles.  The share
// spans few heads: the Q' fragments of up to kHeadsCached heads at a time are
// built in shared memory (fragment order) between two barriers.
//
// As in the full scorer, the 256-long axis is permuted identically for K' and Q'
// so that each thread's 16-byte reads of rows g and g+8 are its A fragments
// (chunks t, t+4, ..., t+28 of the row).  The rows' norms |k'| come from the
// diagonal of the Gram tile K' K'^T, a second set of MMAs on the same fragments,
// instead of 64 scalar multiply-adds per row and thread.  Bound: e = 2^-12 |q'| |k'| / sqrt(d) +
// |s~| 2^-22 + 2^-60 with |q'| = |q|; the modelled tensor-core accumulation error
// of 16 steps of 16 exact products is 272 x 2^-23 ~ 2^-14.9, a 7x margin.
// Optionally carries the copy half of a gather (fetch_copy.cuh).
#include "fetch_copy.cuh"

namespace oasis {

constexpr int kPsWarps = 4;
constexpr int kTileBlocks = 16;
constexpr int kPK = 2 * kD;                             // pooled elements per block
constexpr int kMaxPrefix = 512;                         // requests with an exact tile prefix

// Q' fragment sets held at once: two heads up to 16 query rows, one above (three
// CTAs share an SM's shared memory)
template <int NT>
struct HeadsCached { static constexpr int value = NT <= 2 ? 2 : 1; };

template <int NT>
struct PooledSmem {
  uint2 qf[HeadsCached<NT>::value][NT][8][2][32];  // Q' fragments [head][n-tile][chunk i][half][lane]
  float qn2[2];                                // squared max query norm per cached head
  int pre[kMaxPrefix + 1];                     // tiles before request b (all its KV heads)
};

// positive / negative part of each bf16 of a word pair
__device__ __forceinline__ uint32_t bf2_pos(uint32_t w) {
  const uint32_t m = ((w & 0x8000u) ? 0u : 0xffffu) | ((w & 0x80000000u) ? 0u : 0xffff0000u);
  return w & m;
}
__device__ __forceinline__ uint32_t bf2_neg(uint32_t w) {
  const uint32_t m = ((w & 0x8000u) ? 0xffffu : 0u) | ((w & 0x80000000u) ? 0xffff0000u : 0u);
  return w & m;
}

// Tile sequence of the launch: tile index -> (head, first block of the tile).
struct TileMap {
  const int* pre;   // shared, [B + 1] when exact
  int B, Hkv, nb_max, tpb_nominal;
  bool exact;
  __device__ void locate(int idx, int& head, int& blk0) const {
    if (!exact) {  // every head gets ceil(nb_max / 16) tiles; empty ones are skipped
      head = idx / tpb_nominal;
      blk0 = (idx - head * tpb_nominal) * kTileBlocks;
      return;
    }
    int lo = 0, hi = B - 1;  // the last b with pre[b] <= idx
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (pre[mid] <= idx) lo = mid; else hi = mid - 1;
    }
    const int tb = (pre[lo + 1] - pre[lo]) / Hkv;
    const int local = idx - pre[lo];
    const int h = local / tb;
    head = lo * Hkv + h;
    blk0 = (local - h * tb) * kTileBlocks;
  }
  __device__ int first_tile(int head) const {  // first tile index of `head`
    if (!exact) return head * tpb_nominal;
    const int b = head / Hkv, h = head - b * Hkv;
    return pre[b] + h * ((pre[b + 1] - pre[b]) / Hkv);
  }
};

template <int NT, bool kCopy>
__global__ void __launch_bounds__(kPsWarps * 32, 4)
score_pooled_kernel(Shape s, const uint16_t* __restrict__ kp, const int* __restrict__ ctx_len,
                    const uint16_t* __restrict__ q_la, float2* __restrict__ scores, float inv_sqrt_d, CopyJob job,
                    TraceBuf tb) {
  TraceScope trace_(tb, OASIS_TRACE_SCORE_POOLED);
  constexpr int kHeadsCached = HeadsCached<NT>::value;
  extern __shared__ __align__(128) uint8_t ps_dyn[];
  PooledSmem<NT>& sm = *reinterpret_cast<PooledSmem<NT>*>(ps_dyn);
  uint8_t* copy_base = ps_dyn + ((sizeof(PooledSmem<NT>) + 127) & ~size_t(127));
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int g = lane >> 2, t = lane & 3;
  const long long gwarp = (long long)blockIdx.x * kPsWarps + warp;
  const long long nwarps = (long long)gridDim.x * kPsWarps;
  uint4* copy_buf = reinterpret_cast<uint4*>(copy_base);
  if constexpr (kCopy) copy_begin(job, s, gwarp, nwarps, copy_buf + warp * (kCopyUnitBytes / 16), lane);
  const int G = s.Hq / s.Hkv;
  const int N = s.n_la * G;

  // the tile prefix over requests (every CTA computes the same one)
  TileMap map{sm.pre, s.B, s.Hkv, s.nb_max, (s.nb_max + kTileBlocks - 1) / kTileBlocks, s.B <= kMaxPrefix};
  int total;
  if (map.exact) {
    int run = 0;  // serial over requests in chunks of blockDim.x
    for (int b0 = 0; b0 < s.B; b0 += blockDim.x) {
      const int b = b0 + threadIdx.x;
      const int tiles = b < s.B ? (clamp_nb(ctx_len[b], s.nb_max) + kTileBlocks - 1) / kTileBlocks * s.Hkv : 0;
      // block inclusive scan of `tiles`
      int x = tiles;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      __shared__ int wsum[kPsWarps];
      if (lane == 31) wsum[warp] = x;
      __syncthreads();
      int off = 0;
      for (int w = 0; w < warp; ++w) off += wsum[w];
      int tot = 0;
      for (int w = 0; w < kPsWarps; ++w) tot += wsum[w];
      if (b < s.B) sm.pre[b] = run + off + x - tiles;
      run += tot;
      __syncthreads();
    }
    if (threadIdx.x == 0) sm.pre[s.B] = run;
    __syncthreads();
    total = sm.pre[s.B];
  } else {
    total = s.B * s.Hkv * map.tpb_nominal;
  }
  const int T0 = (int)((long long)blockIdx.x * total / gridDim.x);
  const int T1 = (int)((long long)(blockIdx.x + 1) * total / gridDim.x);
  if (T0 >= T1) {
    if constexpr (kCopy) copy_finish(job, s, gwarp, nwarps, copy_buf + warp * (kCopyUnitBytes / 16), lane);
    return;
  }
  int head_first, head_last, unused;
  map.locate(T0, head_first, unused);
  map.locate(T1 - 1, head_last, unused);

  for (int hg = head_first; hg <= head_last; hg += kHeadsCached) {
    const int nh = min(kHeadsCached, head_last - hg + 1);
    __syncthreads();  // every warp is done with the previous group's fragments
    if (threadIdx.x < 2) sm.qn2[threadIdx.x] = 0.f;
    __syncthreads();
    // this group's share of the tile sequence; warp w takes tiles w, w + 8, ...
    const int g0 = max(T0, map.first_tile(hg));
    const int g1 = hg + nh <= head_last ? min(T1, map.first_tile(hg + nh)) : T1;
    const int ntiles = g0 < g1 ? (g1 - g0 - warp + kPsWarps - 1) / kPsWarps : 0;
    // tile index -> (head slot, first block) without a search: the group's heads
    // own consecutive runs of the sequence starting at ft[0] and ft[1]
    const int ft0 = map.first_tile(hg);
    const int ft1 = nh > 1 ? map.first_tile(hg + 1) : 0x7fffffff;
    const int nbh0 = clamp_nb(ctx_len[hg / s.Hkv], s.nb_max);
    const int nbh1 = nh > 1 ? clamp_nb(ctx_len[(hg + 1) / s.Hkv], s.nb_max) : 0;
    auto where = [&](int idx, int& hs, int& blk0, int& nbv) {
      hs = (kHeadsCached > 1 && idx >= ft1) ? 1 : 0;
      blk0 = (idx - (hs ? ft1 : ft0)) * kTileBlocks;
      nbv = hs ? nbh1 : nbh0;
    };

    // Rolling prefetch: the first tile's loads go out before the Q' fragments are
    // built (they do not depend on them); then, once chunk i of the current tile
    // has fed its MMAs, its registers receive chunk i of this warp's next tile, so
    // a tile's worth of loads stays in flight through the MMAs and the epilogue.
    uint4 ra[8], rb[8];
    int hs_c = 0, blk0_c = 0, nbv_c = 0;
    if (ntiles > 0) {
      where(g0 + warp, hs_c, blk0_c, nbv_c);
      const int blk1 = min(nbv_c, blk0_c + kTileBlocks);
      const uint16_t* base = kp + (long long)(hg + hs_c) * s.nb_max * kPK;
      const int r0 = blk0_c + g, r1 = blk0_c + g + 8;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        ra[i] = r0 < blk1 ? ldg_stream(base + (long long)r0 * kPK + (t + 4 * i) * 8) : make_uint4(0u, 0u, 0u, 0u);
        rb[i] = r1 < blk1 ? ldg_stream(base + (long long)r1 * kPK + (t + 4 * i) * 8) : make_uint4(0u, 0u, 0u, 0u);
      }
    }
    // Q' fragments of the group's heads: warp w builds (head slot, n-tile) pairs w, w + 8, ...
    for (int pair = warp; pair < nh * NT; pair += kPsWarps) {
      const int hs = pair / NT, nt = pair - hs * NT;
      const int head = hg + hs;
      const int b = head / s.Hkv, h = head - b * s.Hkv;
      const int n = nt * 8 + g;
      uint4 v[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) v[i] = make_uint4(0u, 0u, 0u, 0u);
      if (n < N) {
        const int j = n / G, gg = n - j * G;
        const uint16_t* qrow = q_la + (((long long)b * s.n_la + j) * s.Hq + h * G + gg) * kD;
#pragma unroll
        for (int i = 0; i < 4; ++i) v[i] = ldg_nc(qrow + (t + 4 * i) * 8);
      }
      float ss = 0.f;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          ss = fmaf(bf_lo(w[m]), bf_lo(w[m]), ss);
          ss = fmaf(bf_hi(w[m]), bf_hi(w[m]), ss);
        }
        // chunk t + 4i of q' is q+ chunk t + 4i; chunk t + 4(i + 4) is q- chunk t + 4i
        sm.qf[hs][nt][i][0][lane] = make_uint2(bf2_pos(w[0]), bf2_pos(w[1]));
        sm.qf[hs][nt][i][1][lane] = make_uint2(bf2_pos(w[2]), bf2_pos(w[3]));
        sm.qf[hs][nt][i + 4][0][lane] = make_uint2(bf2_neg(w[0]), bf2_neg(w[1]));
        sm.qf[hs][nt][i + 4][1][lane] = make_uint2(bf2_neg(w[2]), bf2_neg(w[3]));
      }
      ss += __shfl_xor_sync(0xffffffffu, ss, 1);
      ss += __shfl_xor_sync(0xffffffffu, ss, 2);
      ss = warp_max(ss);
      // non-negative floats order like their bit patterns
      if (lane == 0) atomicMax(reinterpret_cast<int*>(&sm.qn2[hs]), __float_as_int(ss));
    }
    __syncthreads();

    for (int k = 0; k < ntiles; ++k) {
      const int hs = hs_c, blk0 = blk0_c;
      const int head = hg + hs;
      const int blk1 = min(nbv_c, blk0 + kTileBlocks);
      const int r0 = blk0 + g, r1 = blk0 + g + 8;
      int hs_n = 0, blk0_n = 0, nbv_n = 0;
      if (k + 1 < ntiles) where(g0 + warp + (k + 1) * kPsWarps, hs_n, blk0_n, nbv_n);
      const int blk1_n = min(nbv_n, blk0_n + kTileBlocks);  // 0 when there is no next tile
      const uint16_t* base_n = kp + (long long)(hg + hs_n) * s.nb_max * kPK;
      const int r0n = blk0_n + g, r1n = blk0_n + g + 8;
      const bool ok0 = r0n < blk1_n, ok1 = r1n < blk1_n;
      float acc[NT][4];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
      // |k'|^2 of the 16 rows: the diagonal of the Gram tile K' K'^T, formed on the
      // tensor cores from the A fragments themselves (the B fragment of column n is
      // row n's own A words).  Row r's entry sits in lane 4 (r & 7) + ((r & 7) >> 1).
      // The products are exact and positive, so the fp32 sum is at most 2^-15.9 of
      // itself below the exact one; (1 + 2^-14) makes it an upper bound.
      float gr[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint32_t A[4] = {ra[i].x, ra[i].y, ra[i].z, ra[i].w};
        const uint32_t Bw[4] = {rb[i].x, rb[i].y, rb[i].z, rb[i].w};
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            const uint2 q = sm.qf[hs][nt][i][hh][lane];
            mma_bf16_16816(acc[nt][0], acc[nt][1], acc[nt][2], acc[nt][3], A[2 * hh], Bw[2 * hh], A[2 * hh + 1],
                           Bw[2 * hh + 1], q.x, q.y);
          }
          mma_bf16_16816(gr[0][0], gr[0][1], gr[0][2], gr[0][3], A[2 * hh], Bw[2 * hh], A[2 * hh + 1],
                         Bw[2 * hh + 1], A[2 * hh], A[2 * hh + 1]);
          mma_bf16_16816(gr[1][0], gr[1][1], gr[1][2], gr[1][3], A[2 * hh], Bw[2 * hh], A[2 * hh + 1],
                         Bw[2 * hh + 1], Bw[2 * hh], Bw[2 * hh + 1]);
        }
        ra[i] = ok0 ? ldg_stream(base_n + (long long)r0n * kPK + (t + 4 * i) * 8) : make_uint4(0u, 0u, 0u, 0u);
        rb[i] = ok1 ? ldg_stream(base_n + (long long)r1n * kPK + (t + 4 * i) * 8) : make_uint4(0u, 0u, 0u, 0u);
      }
      hs_c = hs_n;
      blk0_c = blk0_n;
      nbv_c = nbv_n;
      float m0 = neg_inf(), m1 = neg_inf();
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const int n0 = nt * 8 + 2 * t;
        if (n0 < N) { m0 = fmaxf(m0, acc[nt][0]); m1 = fmaxf(m1, acc[nt][2]); }
        if (n0 + 1 < N) { m0 = fmaxf(m0, acc[nt][1]); m1 = fmaxf(m1, acc[nt][3]); }
      }
      m0 = fmaxf(m0, __shfl_xor_sync(0xffffffffu, m0, 1));
      m0 = fmaxf(m0, __shfl_xor_sync(0xffffffffu, m0, 2));
      m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, 1));
      m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, 2));
      const int holder = 4 * g + (g >> 1);
      const float d0 = (g & 1) ? gr[0][1] : gr[0][0];   // row g, column g
      const float d1 = (g & 1) ? gr[1][3] : gr[1][2];   // row g + 8, column g + 8
      const float s0 = __shfl_sync(0xffffffffu, d0, holder) * 1.00006103515625f;  // x (1 + 2^-14)
      const float s1 = __shfl_sync(0xffffffffu, d1, holder) * 1.00006103515625f;
      if (t == 0) {
        const float qnorm = sqrtf(sm.qn2[hs]);
        float2* out = scores + (long long)head * s.nb_max;
        if (r0 < blk1) {
          const float sc = m0 * inv_sqrt_d;
          const float e = kAccRel * 1.0009765625f * qnorm * sqrtf(s0) * inv_sqrt_d +
                          fabsf(sc) * 2.384185791015625e-07f + 8.673617379884035e-19f;
          out[r0] = make_float2(sc, e);
        }
        if (r1 < blk1) {
          const float sc = m1 * inv_sqrt_d;
          const float e = kAccRel * 1.0009765625f * qnorm * sqrtf(s1) * inv_sqrt_d +
                          fabsf(sc) * 2.384185791015625e-07f + 8.673617379884035e-19f;
          out[r1] = make_float2(sc, e);
        }
      }
    }
  }
  if constexpr (kCopy) copy_finish(job, s, gwarp, nwarps, copy_buf + warp * (kCopyUnitBytes / 16), lane);
}

template <int NT, bool kCopy>
static size_t pooled_smem_bytes() {
  return ((sizeof(PooledSmem<NT>) + 127) & ~size_t(127)) + (kCopy ? (size_t)kPsWarps * kCopyUnitBytes : 0);
}

template <int NT, bool kCopy>
static cudaError_t launch_nt2(const Shape& s, const uint16_t* kp, const int* ctx, const uint16_t* q_la,
                              float2* scores, const CopyJob& job, cudaStream_t stream) {
  static int attr_cache[kMaxDevicesCached] = {};
  const size_t smem = pooled_smem_bytes<NT, kCopy>();
  cudaError_t e = ensure_dyn_smem((const void*)score_pooled_kernel<NT, kCopy>, smem, attr_cache);
  if (e != cudaSuccess) return e;
  static int per_sm_cached[kMaxDevicesCached] = {};
  int& per_sm = per_sm_cached[current_device()];
  if (!per_sm) {
    int v = 0;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, score_pooled_kernel<NT, kCopy>, kPsWarps * 32, smem);
    per_sm = v < 1 ? 1 : v;
  }
  const int cap = score_ctas_per_sm_option();
  const int grid = sm_count() * (cap > 0 && cap < per_sm ? cap : per_sm);
  score_pooled_kernel<NT, kCopy><<<grid, kPsWarps * 32, smem, stream>>>(s, kp, ctx, q_la, scores,
                                                                       1.0f / sqrtf((float)s.d), job, trace_buf());
  return cudaGetLastError();
}

template <int NT>
static cudaError_t launch_nt(const Shape& s, const uint16_t* kp, const int* ctx, const uint16_t* q_la,
                             float2* scores, const CopyJob* job, cudaStream_t stream) {
  if (job) return launch_nt2<NT, true>(s, kp, ctx, q_la, scores, *job, stream);
  return launch_nt2<NT, false>(s, kp, ctx, q_la, scores, CopyJob{}, stream);
}

cudaError_t launch_score_pooled(const Shape& s, const uint16_t* kp, const int* ctx, const uint16_t* q_la,
                                float2* scores, const CopyJob* job, cudaStream_t stream) {
  const int NT = (s.n_la * (s.Hq / s.Hkv) + 7) / 8;
  switch (NT) {
    case 1: return launch_nt<1>(s, kp, ctx, q_la, scores, job, stream);
    case 2: return launch_nt<2>(s, kp, ctx, q_la, scores, job, stream);
    case 3: return launch_nt<3>(s, kp, ctx, q_la, scores, job, stream);
    case 4: return launch_nt<4>(s, kp, ctx, q_la, scores, job, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace oasis
