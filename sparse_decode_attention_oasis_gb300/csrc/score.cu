// a1: block scoring against the lookahead queries, on the tensor cores.
//
// score(x) = max over lookahead queries j, GQA query heads g and valid tokens t
// of block x of q_la[j, hG+g] . k_t / sqrt(d)  (OasisKV, metalmedia.ai page,
// Figure 7 caption: the draft queries are compared with the keys to choose the
// blocks the next step needs).
//
// Mapping.  One warp scores one 16-token block at a time as a 16 x N tile
// D = K_blk (16 tok x 128 d) * Q^T (128 d x N queries) with mma.m16n8k16 (bf16
// in, fp32 accumulate).  Because a dot product may sum its d terms in any order,
// the d axis is permuted identically for K and Q: thread (g = lane/4,
// t = lane%4) loads 16-byte chunks t, t+4, t+8, t+12 of token rows g and g+8
// straight from HBM (every 32-byte sector is used by one instruction), and
// those registers are already A fragments.  Q fragments of the head stay in
// registers for the whole run of blocks of that head.
//
// Certified bound.  Each block also gets e >= |s~ - score|: the tensor-core
// fp32 accumulation of 8 steps of 16 exact products is modelled as at most
// 17 truncations of 2^-23 of the running magnitude per step, i.e.
// 136 * 2^-23 ~ 2^-15.9 of sum|q_i k_i| <= |q|_2 |k|_2.  We use 2^-12 (a 15x
// margin), the max query norm of the head and the max key norm of the block
// (computed here in fp32 from the same registers), plus the rounding of the
// 1/sqrt(d) product and an absolute 2^-60 for underflowed products.
//
// With a copy job the kernel also carries the data half of another layer's
// gather (fetch_copy.cuh): every warp stages its first fetched block through
// 8 KiB of shared memory before it starts scoring and writes it to its HBM slot
// afterwards, so the host-link latency overlaps the scoring.
#include "fetch_copy.cuh"

namespace oasis {

constexpr int kScoreWarps = 4;

template <int NT>
struct QFrag {
  uint32_t w[NT][4][4];  // [n-tile][d chunk i][word]
};

// Score blocks [blk0, blk1) of one (request, KV head); the CTA's warps take
// every kScoreWarps-th block.  Query fragments are loaded once per segment.
template <int NT>
__device__ __forceinline__ void score_segment(const Shape& s, const uint16_t* __restrict__ k_hbm,
                                              const uint16_t* __restrict__ q_la, float2* __restrict__ scores,
                                              int b, int h, int ctx, int blk0, int blk1, float inv_sqrt_d,
                                              int warp, int lane) {
  const int g = lane >> 2, t = lane & 3;
  const int G = s.Hq / s.Hkv;
  const int N = s.n_la * G;
  const int head = b * s.Hkv + h;
  const long long T_max = (long long)s.nb_max * kBS;

  // Q fragments: query n = nt*8 + g is lookahead j = n / G, head hG + n % G.
  QFrag<NT> qf;
  float qn2 = 0.f;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int n = nt * 8 + g;
    float ss = 0.f;
    if (n < N) {
      const int j = n / G, gg = n - j * G;
      const uint16_t* qrow = q_la + (((long long)b * s.n_la + j) * s.Hq + h * G + gg) * kD;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        uint4 v = ldg_nc(qrow + (t + 4 * i) * 8);
        qf.w[nt][i][0] = v.x; qf.w[nt][i][1] = v.y; qf.w[nt][i][2] = v.z; qf.w[nt][i][3] = v.w;
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          float a = bf_lo(qf.w[nt][i][m]), bb = bf_hi(qf.w[nt][i][m]);
          ss = fmaf(a, a, ss);
          ss = fmaf(bb, bb, ss);
        }
      }
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int m = 0; m < 4; ++m) qf.w[nt][i][m] = 0u;
    }
    ss += __shfl_xor_sync(0xffffffffu, ss, 1);
    ss += __shfl_xor_sync(0xffffffffu, ss, 2);
    qn2 = fmaxf(qn2, ss);
  }
  qn2 = warp_max(qn2);
  const float qnorm = sqrtf(qn2);

  const uint16_t* kbase = k_hbm + ((long long)head * T_max) * kD;
  int blk = blk0 + warp;
  uint4 ra[4], rb[4];
  if (blk < blk1) {
    const uint16_t* p = kbase + ((long long)blk * kBS) * kD;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      ra[i] = ldg_stream(p + g * kD + (t + 4 * i) * 8);
      rb[i] = ldg_stream(p + (g + 8) * kD + (t + 4 * i) * 8);
    }
  }
  for (; blk < blk1; blk += kScoreWarps) {
    uint4 ca[4], cb[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) { ca[i] = ra[i]; cb[i] = rb[i]; }
    const int nxt = blk + kScoreWarps;
    if (nxt < blk1) {  // prefetch the next block of this warp
      const uint16_t* p = kbase + ((long long)nxt * kBS) * kD;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        ra[i] = ldg_stream(p + g * kD + (t + 4 * i) * 8);
        rb[i] = ldg_stream(p + (g + 8) * kD + (t + 4 * i) * 8);
      }
    }
    float acc[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t A[4] = {ca[i].x, ca[i].y, ca[i].z, ca[i].w};
      const uint32_t Bw[4] = {cb[i].x, cb[i].y, cb[i].z, cb[i].w};
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
          mma_bf16_16816(acc[nt][0], acc[nt][1], acc[nt][2], acc[nt][3], A[2 * hh], Bw[2 * hh],
                         A[2 * hh + 1], Bw[2 * hh + 1], qf.w[nt][i][2 * hh],
                         qf.w[nt][i][2 * hh + 1]);
      }
    }
    const int tok = blk * kBS + g;
    const bool v0 = tok < ctx, v1 = tok + 8 < ctx;
    float m = neg_inf();
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int n0 = nt * 8 + 2 * t;
      if (n0 < N) {
        if (v0) m = fmaxf(m, acc[nt][0]);
        if (v1) m = fmaxf(m, acc[nt][2]);
      }
      if (n0 + 1 < N) {
        if (v0) m = fmaxf(m, acc[nt][1]);
        if (v1) m = fmaxf(m, acc[nt][3]);
      }
    }
    m = warp_max(m);
    // max key norm of the valid tokens of the block
    float s0 = 0.f, s1 = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t A[4] = {ca[i].x, ca[i].y, ca[i].z, ca[i].w};
      const uint32_t Bw[4] = {cb[i].x, cb[i].y, cb[i].z, cb[i].w};
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        float a0 = bf_lo(A[w]), a1 = bf_hi(A[w]);
        float b0 = bf_lo(Bw[w]), b1 = bf_hi(Bw[w]);
        s0 = fmaf(a0, a0, s0); s0 = fmaf(a1, a1, s0);
        s1 = fmaf(b0, b0, s1); s1 = fmaf(b1, b1, s1);
      }
    }
    s0 += __shfl_xor_sync(0xffffffffu, s0, 1);
    s0 += __shfl_xor_sync(0xffffffffu, s0, 2);
    s1 += __shfl_xor_sync(0xffffffffu, s1, 1);
    s1 += __shfl_xor_sync(0xffffffffu, s1, 2);
    float kn2 = fmaxf(v0 ? s0 : 0.f, v1 ? s1 : 0.f);
    kn2 = warp_max(kn2);
    if (lane == 0) {
      const float sc = m * inv_sqrt_d;
      const float e = kAccRel * 1.0009765625f * qnorm * sqrtf(kn2) * inv_sqrt_d +
                      fabsf(sc) * 2.384185791015625e-07f /* 2^-22 */ + 8.673617379884035e-19f /* 2^-60 */;
      scores[(long long)head * s.nb_max + blk] = make_float2(sc, e);
    }
  }
}

// Static work split.  The valid blocks of all heads, request by request and head
// by head within a request, form one sequence; CTA i scores the i-th of gridDim.x
// equal contiguous ranges of it (one or two heads each on the Qwen3-8B decode
// shape), so a batch of ragged contexts loads every CTA alike.  The sequence's
// offsets come from an exclusive prefix over requests of nb(b) * Hkv that every
// CTA computes for itself in shared memory (B <= kMaxPrefix); with more requests
// every head is given nb_max positions and the positions past a head's context
// are skipped.
constexpr int kMaxPrefix = 512;

struct BlockSeq {
  const int* pre;  // shared, [B + 1] when exact
  int Hkv, nb_max, B;
  bool exact;
  // request b, head h and block index of position `idx`, and the end of that head's run
  __device__ void locate(int idx, int& b, int& h, int& blk, int& run_end) const {
    if (!exact) {
      const int head = idx / nb_max;
      b = head / Hkv;
      h = head - b * Hkv;
      blk = idx - head * nb_max;
      run_end = (head + 1) * nb_max;
      return;
    }
    int lo = 0, hi = B - 1;  // the last b with pre[b] <= idx (that request is not empty)
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (pre[mid] <= idx) lo = mid; else hi = mid - 1;
    }
    b = lo;
    const int nbb = (pre[lo + 1] - pre[lo]) / Hkv;
    const int local = idx - pre[lo];
    h = local / nbb;
    blk = local - h * nbb;
    run_end = pre[lo] + (h + 1) * nbb;
  }
};

// kDyn: a share of the sequence of valid blocks is split into equal contiguous
// ranges as in the static kernel (static_permille / 1000 of it); the rest is
// handed out in chunks of `chunk_blocks` positions by an atomic counter
// (work[0]), so thread blocks that start late (their SM still busy with a kernel
// of another stream) take fewer chunks instead of finishing last.  Each block
// claims its next chunk before it scores the current one, so the atomic's latency
// overlaps the scoring.  The last block to finish (work[1] counts them) leaves
// both words at zero for the next launch.
template <int NT, bool kCopy, bool kDyn = false>
__global__ void __launch_bounds__(kScoreWarps * 32, (NT <= 2 ? 4 : 3))
score_blocks_kernel(Shape s, const uint16_t* __restrict__ k_hbm, const int* __restrict__ ctx_len,
                    const uint16_t* __restrict__ q_la, float2* __restrict__ scores, float inv_sqrt_d,
                    CopyJob job, TraceBuf tb, unsigned* __restrict__ work = nullptr, int chunk_blocks = 0,
                    int static_permille = 1000) {
  TraceScope trace_(tb, OASIS_TRACE_SCORE);
  extern __shared__ uint4 copy_buf[];  // [kScoreWarps][512] when kCopy
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const long long gwarp = (long long)blockIdx.x * kScoreWarps + warp;
  const long long nwarps = (long long)gridDim.x * kScoreWarps;
  if constexpr (kCopy) copy_begin(job, s, gwarp, nwarps, copy_buf + warp * (kCopyUnitBytes / 16), lane);

  __shared__ int pre[kMaxPrefix + 1];
  __shared__ int wsum[kScoreWarps];
  __shared__ int dyn_next;
  if constexpr (kDyn) {
    // the first chunk is claimed now; its latency overlaps the prefix and the static share
    if (threadIdx.x == 0) dyn_next = (int)atomicAdd(work, 1u);
  }
  BlockSeq seq{pre, s.Hkv, s.nb_max, s.B, s.B <= kMaxPrefix};
  int total;
  if (seq.exact) {
    int run = 0;
    for (int b0 = 0; b0 < s.B; b0 += kScoreWarps * 32) {
      const int b = b0 + threadIdx.x;
      const int n = b < s.B ? clamp_nb(ctx_len[b], s.nb_max) * s.Hkv : 0;
      int x = n;  // inclusive scan over the CTA
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      if (lane == 31) wsum[warp] = x;
      __syncthreads();
      int off = 0, tot = 0;
#pragma unroll
      for (int w = 0; w < kScoreWarps; ++w) {
        off += w < warp ? wsum[w] : 0;
        tot += wsum[w];
      }
      if (b < s.B) pre[b] = run + off + x - n;
      run += tot;
      __syncthreads();  // wsum is rewritten by the next round
    }
    if (threadIdx.x == 0) pre[s.B] = run;
    __syncthreads();
    total = pre[s.B];
  } else {
    total = s.B * s.Hkv * s.nb_max;
  }
  // score positions [p0, p1) of the sequence: one segment per (request, head) run
  auto run_range = [&](int p0, int p1) {
    for (int pos = p0; pos < p1;) {
      int b, h, blk0, run_end;
      seq.locate(pos, b, h, blk0, run_end);
      const int end = min(p1, run_end);
      const int ctx = ctx_len[b];
      const int blk1 = min(blk0 + (end - pos), clamp_nb(ctx, s.nb_max));
      if (blk0 < blk1) score_segment<NT>(s, k_hbm, q_la, scores, b, h, ctx, blk0, blk1, inv_sqrt_d, warp, lane);
      pos = end;
    }
  };
  const int stat = kDyn ? (int)((long long)total * static_permille / 1000) : total;
  run_range((int)((long long)blockIdx.x * stat / gridDim.x), (int)((long long)(blockIdx.x + 1) * stat / gridDim.x));
  if constexpr (kDyn) {
    __syncthreads();  // dyn_next is visible
    int chunk = dyn_next;
    for (;;) {
      const long long c0 = stat + (long long)chunk * chunk_blocks;
      if (c0 >= total) break;
      __syncthreads();  // every thread has read dyn_next
      if (threadIdx.x == 0) dyn_next = (int)atomicAdd(work, 1u);  // the next chunk, claimed ahead
      run_range((int)c0, (int)min((long long)total, c0 + chunk_blocks));
      __syncthreads();
      chunk = dyn_next;
    }
    if (threadIdx.x == 0) {
      __threadfence();  // this block's last claim is ordered before its count
      if (atomicAdd(work + 1, 1u) == gridDim.x - 1) {  // every block has claimed past the end
        work[0] = 0u;
        work[1] = 0u;
      }
    }
  }
  if constexpr (kCopy) copy_finish(job, s, gwarp, nwarps, copy_buf + warp * (kCopyUnitBytes / 16), lane);
}

int score_grid_limit(int nt);

constexpr int kScoreCopySmem = kScoreWarps * kCopyUnitBytes;  // 32 KiB

template <bool kCopy>
static cudaError_t launch_score(const Shape& s, const uint16_t* k, const int* ctx, const uint16_t* q_la,
                                float2* scores, const CopyJob& job, cudaStream_t stream) {
  const int N = s.n_la * (s.Hq / s.Hkv);
  const int NT = (N + 7) / 8;
  const float inv = 1.0f / sqrtf((float)s.d);
  // at least kMinBlocksPerCta positions of the sequence per CTA; the copy wants a
  // warp for each live fetch entry, so its grid is never cut to the work
  constexpr long long kMinBlocksPerCta = 4 * kScoreWarps;
  const long long positions = (long long)s.B * s.Hkv * s.nb_max;
  const long long by_work = (positions + kMinBlocksPerCta - 1) / kMinBlocksPerCta;
  const int limit = score_grid_limit(NT);
  int grid = kCopy || by_work >= limit ? limit : (int)by_work;
  if (grid < 1) grid = 1;
  const dim3 block(kScoreWarps * 32);
  const size_t smem = kCopy ? kScoreCopySmem : 0;
  const TraceBuf tb = trace_buf();
  switch (NT) {
    case 1: score_blocks_kernel<1, kCopy><<<grid, block, smem, stream>>>(s, k, ctx, q_la, scores, inv, job, tb); break;
    case 2: score_blocks_kernel<2, kCopy><<<grid, block, smem, stream>>>(s, k, ctx, q_la, scores, inv, job, tb); break;
    case 3: score_blocks_kernel<3, kCopy><<<grid, block, smem, stream>>>(s, k, ctx, q_la, scores, inv, job, tb); break;
    case 4: score_blocks_kernel<4, kCopy><<<grid, block, smem, stream>>>(s, k, ctx, q_la, scores, inv, job, tb); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

// The dynamic variant: chunks of 64 blocks from an atomic counter; the grid leaves
// `reserve` thread-block slots of the GPU free for kernels on other streams.
cudaError_t launch_score_blocks_dyn(const Shape& s, const uint16_t* k, const int* ctx, const uint16_t* q_la,
                                    float2* scores, unsigned* work, int reserve, cudaStream_t stream) {
  const int N = s.n_la * (s.Hq / s.Hkv);
  const int NT = (N + 7) / 8;
  constexpr int kDynChunk = 64;
  const long long total = (long long)s.B * s.Hkv * ((s.nb_max + kDynChunk - 1) / kDynChunk);
  const int share = score_static_share_option();
  const float inv = 1.0f / sqrtf((float)s.d);
  int grid = score_grid_limit(NT) - reserve;
  if (grid > total) grid = (int)total;
  if (grid < 1) grid = 1;
  const dim3 block(kScoreWarps * 32);
  const CopyJob job{};
  const TraceBuf tb = trace_buf();
  switch (NT) {
    case 1: score_blocks_kernel<1, false, true><<<grid, block, 0, stream>>>(s, k, ctx, q_la, scores, inv, job, tb, work, kDynChunk, share); break;
    case 2: score_blocks_kernel<2, false, true><<<grid, block, 0, stream>>>(s, k, ctx, q_la, scores, inv, job, tb, work, kDynChunk, share); break;
    case 3: score_blocks_kernel<3, false, true><<<grid, block, 0, stream>>>(s, k, ctx, q_la, scores, inv, job, tb, work, kDynChunk, share); break;
    case 4: score_blocks_kernel<4, false, true><<<grid, block, 0, stream>>>(s, k, ctx, q_la, scores, inv, job, tb, work, kDynChunk, share); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t launch_score_blocks(const Shape& s, const uint16_t* k, const int* ctx, const uint16_t* q_la,
                                float2* scores, cudaStream_t stream) {
  return launch_score<false>(s, k, ctx, q_la, scores, CopyJob{}, stream);
}

cudaError_t launch_score_blocks_copy(const Shape& s, const uint16_t* k, const int* ctx, const uint16_t* q_la,
                                     float2* scores, const CopyJob& job, cudaStream_t stream) {
  return launch_score<true>(s, k, ctx, q_la, scores, job, stream);
}

int score_grid_limit(int nt) {
  static int per_sm_cached[kMaxDevicesCached][5] = {};
  const int dev = current_device();
  int& per_sm = per_sm_cached[dev][nt];
  if (!per_sm) {
    const int threads = kScoreWarps * 32;
    int v = 0;
    switch (nt) {
      case 1: cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, score_blocks_kernel<1, false>, threads, 0); break;
      case 2: cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, score_blocks_kernel<2, false>, threads, 0); break;
      case 3: cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, score_blocks_kernel<3, false>, threads, 0); break;
      default: cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, score_blocks_kernel<4, false>, threads, 0); break;
    }
    per_sm = v < 1 ? 1 : v;
  }
  // a caller that runs other kernels beside the scorer can ask for fewer CTAs per SM
  const int cap = score_ctas_per_sm_option();
  return sm_count() * (cap > 0 && cap < per_sm ? cap : per_sm);
}

}  // namespace oasis
