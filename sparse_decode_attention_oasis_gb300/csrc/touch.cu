// One read of a page-locked, device-mapped host range through the SMs' load path.
//
// On the GB300 systems this library was measured on, the first zero-copy reads
// that SMs make into some regions of a large pinned host allocation stall for
// milliseconds (repeatedly, until the region has been read); copy-engine
// transfers do not clear the condition, SM loads do.  A gather that meets such a
// stall holds up its whole decode step, so a caller that has just filled the
// host tier can read it once with this kernel, off the latency-critical path.
// Every 16-byte piece is loaded (grid-stride, 8 loads in flight per thread); the
// values are folded into a word that is written out only if it equals a value
// that cannot occur, so the loads are kept without writing anything.
#include "common.cuh"

namespace oasis {

constexpr int kTouchThreads = 256;
constexpr int kTouchUnroll = 8;

__global__ void __launch_bounds__(kTouchThreads)
touch_host_kernel(const uint4* __restrict__ p, unsigned long long n16, unsigned* __restrict__ sink) {
  const unsigned long long stride = (unsigned long long)gridDim.x * blockDim.x;
  unsigned acc = 0u;
  unsigned long long i = (unsigned long long)blockIdx.x * blockDim.x + threadIdx.x;
  for (; i + (kTouchUnroll - 1) * stride < n16; i += kTouchUnroll * stride) {
    uint4 v[kTouchUnroll];
#pragma unroll
    for (int u = 0; u < kTouchUnroll; ++u) {
      asm volatile("ld.global.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                   : "=r"(v[u].x), "=r"(v[u].y), "=r"(v[u].z), "=r"(v[u].w)
                   : "l"(p + i + u * stride));
    }
#pragma unroll
    for (int u = 0; u < kTouchUnroll; ++u) acc ^= v[u].x ^ v[u].y ^ v[u].z ^ v[u].w;
  }
  for (; i < n16; i += stride) {
    uint4 v;
    asm volatile("ld.global.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p + i));
    acc ^= v.x ^ v.y ^ v.z ^ v.w;
  }
  if (acc == 0x9e3779b9u && sink) *sink = acc;  // keeps the loads; practically never taken
}

cudaError_t launch_touch_host(const void* dev_ptr, size_t bytes, unsigned* sink, cudaStream_t stream) {
  const unsigned long long n16 = bytes / 16;
  if (n16 == 0) return cudaSuccess;
  long long grid = 8LL * sm_count();
  const long long need = (long long)((n16 + kTouchThreads - 1) / kTouchThreads);
  if (grid > need) grid = need;
  touch_host_kernel<<<(unsigned)grid, kTouchThreads, 0, stream>>>(static_cast<const uint4*>(dev_ptr), n16, sink);
  return cudaGetLastError();
}

}  // namespace oasis
