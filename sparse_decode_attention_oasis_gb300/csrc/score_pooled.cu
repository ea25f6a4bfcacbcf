// f1: block scoring from the min/max pooled keys, on the tensor cores.
//
// metalmedia.ai page, Figure 7 caption: the draft query scans the compressed
// (per-block min/max pooled) keys to predict the next step's top-K blocks.
// With hi/lo the pooled rows of block x, the pooled score of query n is the
// largest q.k any key inside the box [lo, hi] can reach:
//   P_n(x) = sum_i max(q_i hi_i, q_i lo_i) = sum_i q+_i hi_i + sum_i q-_i lo_i,
// q+ = max(q, 0), q- = min(q, 0) (lo <= hi).  So P_n(x) = q'.k' with
// q' = [q+ | q-] and k' = [hi | lo], a 256-long dot product, and a block is ONE
// 256-element row: one warp scores 16 blocks as a 16 x N tile
// D = K' (16 x 256) * Q'^T (256 x N) with mma.m16n8k16 (bf16 in, fp32 accumulate).
// score(x) = max over lookahead j and group heads g of P / sqrt(d).  The reads are
// 512 bytes per block instead of 4 KiB.
//
// As in the full scorer, the 256-long axis is permuted identically for K' and Q'
// so that each thread's 16-byte loads of rows g and g+8 are its A fragments
// (chunks t, t+4, ..., t+28 of the row).  Each CTA takes a contiguous range of
// chunks of 128 blocks; Q' fragments are built in shared memory (fragment order,
// conflict-free) whenever that range moves to another head.  Bound: e = 2^-12 |q'|
// |k'| / sqrt(d) + |s~| 2^-22 + 2^-60 with |q'| = |q|; the modelled tensor-core
// accumulation error of 16 steps of 16 exact products is 272 x 2^-23 ~ 2^-14.9,
// a 7x margin.  Optionally carries the copy half of a gather (fetch_copy.cuh).
#include "fetch_copy.cuh"

namespace oasis {

constexpr int kPsWarps = 4;
constexpr int kPsChunk = 128;  // blocks per (CTA, head) work item
constexpr int kPK = 2 * kD;    // pooled elements per block

// positive / negative part of each bf16 of a word pair
__device__ __forceinline__ uint32_t bf2_pos(uint32_t w) {
  const uint32_t m = ((w & 0x8000u) ? 0u : 0xffffu) | ((w & 0x80000000u) ? 0u : 0xffff0000u);
  return w & m;
}
__device__ __forceinline__ uint32_t bf2_neg(uint32_t w) {
  const uint32_t m = ((w & 0x8000u) ? 0xffffu : 0u) | ((w & 0x80000000u) ? 0xffff0000u : 0u);
  return w & m;
}

template <int NT, bool kCopy>
__global__ void __launch_bounds__(kPsWarps * 32, 3)
score_pooled_kernel(Shape s, const uint16_t* __restrict__ kp, const int* __restrict__ ctx_len,
                    const uint16_t* __restrict__ q_la, float2* __restrict__ scores, int chunks_per_head,
                    int total_chunks, float inv_sqrt_d, CopyJob job) {
  __shared__ uint2 qf[NT][8][2][32];  // Q' fragments [n-tile][chunk i][half][lane]
  __shared__ float qn_w[kPsWarps];
  extern __shared__ uint4 copy_buf[];  // [kPsWarps][512] when kCopy
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int g = lane >> 2, t = lane & 3;
  const long long gwarp = (long long)blockIdx.x * kPsWarps + warp;
  const long long nwarps = (long long)gridDim.x * kPsWarps;
  if constexpr (kCopy) copy_begin(job, s, gwarp, nwarps, copy_buf + warp * (kCopyUnitBytes / 16), lane);
  const int G = s.Hq / s.Hkv;
  const int N = s.n_la * G;

  // a contiguous range of chunks per CTA: consecutive chunks mostly share a head,
  // so the Q' fragments are rebuilt only when the head changes
  const int c_begin = (int)((long long)blockIdx.x * total_chunks / gridDim.x);
  const int c_end = (int)((long long)(blockIdx.x + 1) * total_chunks / gridDim.x);
  int cur_head = -1;
  float qnorm = 0.f;
  for (int chunk = c_begin; chunk < c_end; ++chunk) {
    const int head = chunk / chunks_per_head;
    const int c = chunk - head * chunks_per_head;
    const int b = head / s.Hkv, h = head - b * s.Hkv;
    const int nb = clamp_nb(ctx_len[b], s.nb_max);
    const int blk0 = c * kPsChunk;
    if (blk0 >= nb) continue;
    const int blk1 = min(nb, blk0 + kPsChunk);
    if (head != cur_head) {
    cur_head = head;
    __syncthreads();  // every warp is done with the previous head's fragments
    float qn2 = 0.f;
    for (int nt = warp; nt < NT; nt += kPsWarps) {
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
        qf[nt][i][0][lane] = make_uint2(bf2_pos(w[0]), bf2_pos(w[1]));
        qf[nt][i][1][lane] = make_uint2(bf2_pos(w[2]), bf2_pos(w[3]));
        qf[nt][i + 4][0][lane] = make_uint2(bf2_neg(w[0]), bf2_neg(w[1]));
        qf[nt][i + 4][1][lane] = make_uint2(bf2_neg(w[2]), bf2_neg(w[3]));
      }
      ss += __shfl_xor_sync(0xffffffffu, ss, 1);
      ss += __shfl_xor_sync(0xffffffffu, ss, 2);
      qn2 = fmaxf(qn2, ss);
    }
    qn2 = warp_max(qn2);
    if (lane == 0) qn_w[warp] = qn2;
    __syncthreads();
    float qmax = qn_w[0];
#pragma unroll
    for (int w = 1; w < kPsWarps; ++w) qmax = fmaxf(qmax, qn_w[w]);
    qnorm = sqrtf(qmax);
    }

    const uint16_t* base = kp + (long long)head * s.nb_max * kPK;
    for (int tile = blk0 + warp * 16; tile < blk1; tile += kPsWarps * 16) {
      const int r0 = tile + g, r1 = tile + g + 8;
      uint4 ra[8], rb[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        ra[i] = r0 < blk1 ? ldg_stream(base + (long long)r0 * kPK + (t + 4 * i) * 8) : make_uint4(0u, 0u, 0u, 0u);
        rb[i] = r1 < blk1 ? ldg_stream(base + (long long)r1 * kPK + (t + 4 * i) * 8) : make_uint4(0u, 0u, 0u, 0u);
      }
      float acc[NT][4];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint32_t A[4] = {ra[i].x, ra[i].y, ra[i].z, ra[i].w};
        const uint32_t Bw[4] = {rb[i].x, rb[i].y, rb[i].z, rb[i].w};
#pragma unroll
        for (int hh = 0; hh < 2; ++hh)
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            const uint2 q = qf[nt][i][hh][lane];
            mma_bf16_16816(acc[nt][0], acc[nt][1], acc[nt][2], acc[nt][3], A[2 * hh], Bw[2 * hh], A[2 * hh + 1],
                           Bw[2 * hh + 1], q.x, q.y);
          }
      }
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
      float s0 = 0.f, s1 = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint32_t A[4] = {ra[i].x, ra[i].y, ra[i].z, ra[i].w};
        const uint32_t Bw[4] = {rb[i].x, rb[i].y, rb[i].z, rb[i].w};
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          s0 = fmaf(bf_lo(A[w]), bf_lo(A[w]), s0); s0 = fmaf(bf_hi(A[w]), bf_hi(A[w]), s0);
          s1 = fmaf(bf_lo(Bw[w]), bf_lo(Bw[w]), s1); s1 = fmaf(bf_hi(Bw[w]), bf_hi(Bw[w]), s1);
        }
      }
      s0 += __shfl_xor_sync(0xffffffffu, s0, 1);
      s0 += __shfl_xor_sync(0xffffffffu, s0, 2);
      s1 += __shfl_xor_sync(0xffffffffu, s1, 1);
      s1 += __shfl_xor_sync(0xffffffffu, s1, 2);
      if (t == 0) {
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

template <int NT>
static int pooled_grid_limit() {
  static int per_sm_cached[kMaxDevicesCached] = {};
  const int dev = current_device();
  int& per_sm = per_sm_cached[dev];
  if (!per_sm) {
    int v = 0;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, score_pooled_kernel<NT, false>, kPsWarps * 32, 0);
    per_sm = v < 1 ? 1 : v;
  }
  const int cap = score_ctas_per_sm_option();
  return sm_count() * (cap > 0 && cap < per_sm ? cap : per_sm);
}

template <int NT>
static cudaError_t launch_nt(const Shape& s, const uint16_t* kp, const int* ctx, const uint16_t* q_la,
                             float2* scores, const CopyJob* job, cudaStream_t stream) {
  const int chunks_per_head = (s.nb_max + kPsChunk - 1) / kPsChunk;
  const int total = s.B * s.Hkv * chunks_per_head;
  const float inv = 1.0f / sqrtf((float)s.d);
  const int lim = pooled_grid_limit<NT>();
  if (job) {
    static int attr_cache[kMaxDevicesCached] = {};
    cudaError_t e = ensure_dyn_smem((const void*)score_pooled_kernel<NT, true>, kPsWarps * kCopyUnitBytes, attr_cache);
    if (e != cudaSuccess) return e;
    score_pooled_kernel<NT, true><<<lim, kPsWarps * 32, kPsWarps * kCopyUnitBytes, stream>>>(
        s, kp, ctx, q_la, scores, chunks_per_head, total, inv, *job);
  } else {
    const int grid = max(1, min(total, lim));
    score_pooled_kernel<NT, false><<<grid, kPsWarps * 32, 0, stream>>>(s, kp, ctx, q_la, scores, chunks_per_head,
                                                                        total, inv, CopyJob{});
  }
  return cudaGetLastError();
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
