// Device helpers shared by the sm_103a kernels of the lookahead sparse decode path.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/oasis.h"

namespace oasis {

constexpr int kD = 128;   // head dimension
constexpr int kBS = 16;   // tokens per block
__device__ __forceinline__ float neg_inf() { return __int_as_float(0xff800000); }

// Relative accumulation bound used for tensor-core block scores (see score.cu).
constexpr float kAccRel = 1.0f / 4096.0f;  // 2^-12

struct Shape {
  int B, Hq, Hkv, d, bs, nb_max, n_la, Kb, P;
  __host__ __device__ int G() const { return Hq / Hkv; }
  __host__ __device__ int N() const { return n_la * (Hq / Hkv); }
  __host__ __device__ long long T_max() const { return (long long)nb_max * bs; }
};

__device__ __forceinline__ int clamp_nb(int ctx, int nb_max) {
  if (ctx <= 0) return 0;
  int nb = (ctx + kBS - 1) / kBS;
  return nb < nb_max ? nb : nb_max;
}

// 16-byte streaming load that skips L1 allocation.
__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__device__ __forceinline__ uint4 ldg_nc(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// bf16x2 word -> two floats (exact).
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// D += A(16x16, row) * B(16x8, col), bf16 inputs, fp32 accumulators.
__device__ __forceinline__ void mma_bf16_16816(float& c0, float& c1, float& c2, float& c3,
                                               uint32_t a0, uint32_t a1, uint32_t a2,
                                               uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c0), "+f"(c1), "+f"(c2), "+f"(c3)
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Pack two floats into a bf16x2 word (round to nearest even); lo in bits 0..15.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Order-preserving map float -> uint32 (larger float -> larger key); -0 < +0.
__device__ __forceinline__ uint32_t float_key(float f) {
  uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_float(uint32_t k) {
  uint32_t u = (k & 0x80000000u) ? (k & 0x7fffffffu) : ~k;
  return __uint_as_float(u);
}

// Process-wide launch option set by oasis_set_option (0 = the kernel's own choice).
int score_ctas_per_sm_option();
int copy_ctas_option();
int score_static_share_option();  // per mille of the valid blocks in fixed shares (dynamic scorer)

// Kernel span trace (oasis_trace_set): passed by value to every traced kernel;
// ctl == nullptr when tracing is off.
struct TraceBuf {
  unsigned* ctl;            // [2 * OASIS_TRACE_KINDS]: records begun, blocks finished, per kind
  unsigned long long* rec;  // [OASIS_TRACE_KINDS][cap][2]: ~earliest start, latest end (ns)
  int cap;
};
TraceBuf trace_buf();  // the buffer set now (host)

__device__ __forceinline__ unsigned long long trace_now() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// One object per thread block, first statement of a traced kernel: thread 0 reads
// the timer and the kind's record index when the block starts and folds its start
// and end into that record when the block ends (any return); the last block of
// the launch to finish moves the kind on to the next record.  Launches of one
// kind that are stream-ordered read distinct indices: every block of the earlier
// launch has finished, index advanced, before any block of the later one starts.
struct TraceScope {
  unsigned* ctl;
  unsigned long long* rec;
  int cap, kind;
  unsigned long long t0 = 0;
  unsigned seq = 0;
  __device__ __forceinline__ TraceScope(const TraceBuf& b, int k) : ctl(b.ctl), rec(b.rec), cap(b.cap), kind(k) {
    if (ctl != nullptr && threadIdx.x == 0 && threadIdx.y == 0 && threadIdx.z == 0) {
      t0 = trace_now();
      seq = *reinterpret_cast<volatile unsigned*>(ctl + 2 * kind);
    }
  }
  __device__ __forceinline__ ~TraceScope() {
    if (ctl != nullptr && threadIdx.x == 0 && threadIdx.y == 0 && threadIdx.z == 0) {
      const unsigned long long t1 = trace_now();
      unsigned long long* r = rec + ((long long)kind * cap + (long long)(seq % (unsigned)cap)) * 2;
      atomicMax(r, ~t0);
      atomicMax(r + 1, t1);
      __threadfence();
      const unsigned blocks = gridDim.x * gridDim.y * gridDim.z;
      if (atomicAdd(ctl + 2 * kind + 1, 1u) == blocks - 1) {
        ctl[2 * kind + 1] = 0u;
        __threadfence();
        atomicAdd(ctl + 2 * kind, 1u);
      }
    }
  }
};

// Host-side caches so that a launch costs no more than the launch itself.
constexpr int kMaxDevicesCached = 64;

inline int current_device() {
  int dev = 0;
  cudaGetDevice(&dev);
  return dev < 0 || dev >= kMaxDevicesCached ? 0 : dev;
}

inline int sm_count() {
  static int cached[kMaxDevicesCached] = {};
  const int dev = current_device();
  if (!cached[dev]) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cached[dev] = n > 0 ? n : 1;
  }
  return cached[dev];
}

// Raise a kernel's dynamic shared-memory limit once per device (and when a larger
// size is needed); `cache` is that kernel's per-device record.
inline cudaError_t ensure_dyn_smem(const void* fn, size_t bytes, int* cache) {
  const int dev = current_device();
  if (cache[dev] >= (int)bytes) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e == cudaSuccess) cache[dev] = (int)bytes;
  return e;
}

}  // namespace oasis
