// Appending each request's newly decoded token to the key cache, the host tier
// and, when its block is resident, to the block's HBM slot.
//
// Decode grows the KV cache by one token per request per step (OasisKV abstract:
// the KV cache dominates memory footprint and traffic during token generation;
// metalmedia.ai page, Table 1 "long output" and Figure 11 caption, requests that
// generate thousands of tokens).  The block that receives the token stays
// coherent in all three places, so scoring, the gather and attention all see it.
//
// One thread block per request: for every KV head, 16 threads move the token's
// 256-byte key and value rows with 16-byte stores (the host-tier stores are
// zero-copy writes over the host link); then, when asked, ctx_len[b] is advanced.
#include "common.cuh"

namespace oasis {

constexpr int kAppendThreads = 128;

__global__ void __launch_bounds__(kAppendThreads)
append_kv_kernel(Shape s, const uint16_t* __restrict__ k_new, const uint16_t* __restrict__ v_new,
                 int* __restrict__ ctx_len, uint16_t* __restrict__ k_hbm, uint16_t* __restrict__ host_kv,
                 const int* __restrict__ blk2slot, uint16_t* __restrict__ k_pool, uint16_t* __restrict__ v_pool,
                 int advance, unsigned* __restrict__ err, TraceBuf tb) {
  TraceScope trace_(tb, OASIS_TRACE_APPEND);
  const int b = blockIdx.x;
  const int t = ctx_len[b];
  const long long T_max = (long long)s.nb_max * kBS;
  if (t < 0 || t >= T_max) {
    if (threadIdx.x == 0 && err) atomicOr(err, OASIS_EW_BAD_COUNT);
    return;
  }
  const int blk = t / kBS, r = t - blk * kBS;
  for (int i = threadIdx.x; i < s.Hkv * 16; i += blockDim.x) {
    const int h = i >> 4, c = i & 15;
    const long long head = (long long)b * s.Hkv + h;
    const uint4 kv = reinterpret_cast<const uint4*>(k_new + head * kD)[c];
    const uint4 vv = reinterpret_cast<const uint4*>(v_new + head * kD)[c];
    reinterpret_cast<uint4*>(k_hbm + (head * T_max + t) * kD)[c] = kv;
    uint16_t* unit = host_kv + (head * s.nb_max + blk) * (2 * kBS * kD);
    reinterpret_cast<uint4*>(unit + r * kD)[c] = kv;
    reinterpret_cast<uint4*>(unit + (kBS + r) * kD)[c] = vv;
    const int slot = blk2slot[head * s.nb_max + blk];
    if (slot >= s.P) {
      if (err) atomicOr(err, OASIS_EW_BAD_SLOT);
    } else if (slot >= 0) {
      reinterpret_cast<uint4*>(k_pool + ((head * s.P + slot) * kBS + r) * kD)[c] = kv;
      reinterpret_cast<uint4*>(v_pool + ((head * s.P + slot) * kBS + r) * kD)[c] = vv;
    }
  }
  if (!advance) return;
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence_system();
    ctx_len[b] = t + 1;
  }
}

cudaError_t launch_append_kv(const Shape& s, const uint16_t* k_new, const uint16_t* v_new, int* ctx,
                             uint16_t* k_hbm, uint16_t* host_kv, const int* blk2slot, uint16_t* k_pool,
                             uint16_t* v_pool, int advance, unsigned* err, cudaStream_t stream) {
  append_kv_kernel<<<s.B, kAppendThreads, 0, stream>>>(s, k_new, v_new, ctx, k_hbm, host_kv, blk2slot, k_pool,
                                                       v_pool, advance, err, trace_buf());
  return cudaGetLastError();
}

}  // namespace oasis
