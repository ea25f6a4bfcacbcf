// f1: per-block min/max pooling of the keys into the compressed key cache, and
// its update when a decoded token is appended.
//
// metalmedia.ai page, Figure 7 caption (left): besides the sparse working set,
// the GPU keeps compressed keys made by per-block min/max pooling, and the draft
// query scans those instead of the full keys.  For block x of a head:
//   hi[x][i] = max over the valid tokens t of x (t < ctx) of k[t][i], lo the min;
// blocks without a valid token hold zeros.  The max or min of bf16 values is one
// of them, so the cache is exact.  Layout bf16 [B][Hkv][nb_max][2][d]: the hi
// row then the lo row, 512 bytes per block (an eighth of the block's keys).
//
// Pooling: one warp per block; lane l owns dims 4l..4l+3 and walks the block's
// valid rows with 8-byte loads (each row read is one 256-byte coalesced access).
#include "common.cuh"

namespace oasis {

constexpr int kPoolThreads = 256;

__device__ __forceinline__ void bf4_to_f(uint2 v, float* f) {
  f[0] = bf_lo(v.x); f[1] = bf_hi(v.x); f[2] = bf_lo(v.y); f[3] = bf_hi(v.y);
}

__device__ __forceinline__ uint16_t f_to_bf_exact(float f) { return (uint16_t)(__float_as_uint(f) >> 16); }

__global__ void __launch_bounds__(kPoolThreads)
pool_keys_kernel(Shape s, const uint16_t* __restrict__ k_hbm, const int* __restrict__ ctx_len,
                 uint16_t* __restrict__ kpooled) {
  const int lane = threadIdx.x & 31;
  const long long w = ((long long)blockIdx.x * kPoolThreads + threadIdx.x) >> 5;
  const long long total = (long long)s.B * s.Hkv * s.nb_max;
  if (w >= total) return;
  const long long head = w / s.nb_max;
  const int x = (int)(w - head * s.nb_max);
  const int b = (int)(head / s.Hkv);
  const int ctx = ctx_len[b];
  const int t0 = x * kBS;
  const int nv = ctx <= t0 ? 0 : min(kBS, ctx - t0);
  uint2 ho = make_uint2(0u, 0u), lo = make_uint2(0u, 0u);
  if (nv > 0) {
    const uint16_t* rows = k_hbm + ((head * s.nb_max + x) * kBS) * kD + lane * 4;
    float mx[4], mn[4];
    bf4_to_f(*reinterpret_cast<const uint2*>(rows), mx);
#pragma unroll
    for (int i = 0; i < 4; ++i) mn[i] = mx[i];
    for (int r = 1; r < nv; ++r) {
      float v[4];
      bf4_to_f(*reinterpret_cast<const uint2*>(rows + r * kD), v);
#pragma unroll
      for (int i = 0; i < 4; ++i) { mx[i] = fmaxf(mx[i], v[i]); mn[i] = fminf(mn[i], v[i]); }
    }
    ho.x = f_to_bf_exact(mx[0]) | ((uint32_t)f_to_bf_exact(mx[1]) << 16);
    ho.y = f_to_bf_exact(mx[2]) | ((uint32_t)f_to_bf_exact(mx[3]) << 16);
    lo.x = f_to_bf_exact(mn[0]) | ((uint32_t)f_to_bf_exact(mn[1]) << 16);
    lo.y = f_to_bf_exact(mn[2]) | ((uint32_t)f_to_bf_exact(mn[3]) << 16);
  }
  uint16_t* out = kpooled + w * (2 * kD) + lane * 4;
  *reinterpret_cast<uint2*>(out) = ho;
  *reinterpret_cast<uint2*>(out + kD) = lo;
}

// Fold each request's new key (written at token position ctx_len[b]) into its
// block's pooled rows: a block's first token sets both rows.
__global__ void __launch_bounds__(kPoolThreads)
pool_append_kernel(Shape s, const uint16_t* __restrict__ k_new, const int* __restrict__ ctx_len,
                   uint16_t* __restrict__ kpooled, unsigned* __restrict__ err) {
  const int lane = threadIdx.x & 31;
  const long long head = ((long long)blockIdx.x * kPoolThreads + threadIdx.x) >> 5;
  if (head >= (long long)s.B * s.Hkv) return;
  const int b = (int)(head / s.Hkv);
  const int t = ctx_len[b];
  if (t < 0 || t >= s.nb_max * kBS) {
    if (lane == 0 && err) atomicOr(err, OASIS_EW_BAD_COUNT);
    return;
  }
  const int x = t / kBS;
  uint16_t* row = kpooled + (head * s.nb_max + x) * (2 * kD) + lane * 4;
  float v[4];
  bf4_to_f(*reinterpret_cast<const uint2*>(k_new + head * kD + lane * 4), v);
  float mx[4], mn[4];
  if (t % kBS == 0) {
#pragma unroll
    for (int i = 0; i < 4; ++i) mx[i] = mn[i] = v[i];
  } else {
    bf4_to_f(*reinterpret_cast<const uint2*>(row), mx);
    bf4_to_f(*reinterpret_cast<const uint2*>(row + kD), mn);
#pragma unroll
    for (int i = 0; i < 4; ++i) { mx[i] = fmaxf(mx[i], v[i]); mn[i] = fminf(mn[i], v[i]); }
  }
  uint2 ho, lo;
  ho.x = f_to_bf_exact(mx[0]) | ((uint32_t)f_to_bf_exact(mx[1]) << 16);
  ho.y = f_to_bf_exact(mx[2]) | ((uint32_t)f_to_bf_exact(mx[3]) << 16);
  lo.x = f_to_bf_exact(mn[0]) | ((uint32_t)f_to_bf_exact(mn[1]) << 16);
  lo.y = f_to_bf_exact(mn[2]) | ((uint32_t)f_to_bf_exact(mn[3]) << 16);
  *reinterpret_cast<uint2*>(row) = ho;
  *reinterpret_cast<uint2*>(row + kD) = lo;
}

cudaError_t launch_pool_keys(const Shape& s, const uint16_t* k, const int* ctx, uint16_t* kpooled,
                             cudaStream_t stream) {
  const long long warps = (long long)s.B * s.Hkv * s.nb_max;
  const long long grid = (warps * 32 + kPoolThreads - 1) / kPoolThreads;
  pool_keys_kernel<<<(unsigned)grid, kPoolThreads, 0, stream>>>(s, k, ctx, kpooled);
  return cudaGetLastError();
}

cudaError_t launch_pool_append(const Shape& s, const uint16_t* k_new, const int* ctx, uint16_t* kpooled,
                               unsigned* err, cudaStream_t stream) {
  const long long warps = (long long)s.B * s.Hkv;
  const long long grid = (warps * 32 + kPoolThreads - 1) / kPoolThreads;
  pool_append_kernel<<<(unsigned)grid, kPoolThreads, 0, stream>>>(s, k_new, ctx, kpooled, err);
  return cudaGetLastError();
}

}  // namespace oasis
