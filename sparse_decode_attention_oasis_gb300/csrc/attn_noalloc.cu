// Allocation-free variant of the sparse decode attention call.
//
// Some callers cannot hand the library a device workspace: a serving loop that
// fixes its device-memory budget at start-up and forbids any later allocation,
// or host code that must not call cudaMalloc on its decode path because the
// call can block on the device.  For them this entry point runs the same two
// attention kernels with their split-K scratch in a file-scope device array
// instead of a caller buffer.  The array (OASIS_ATTN_NOALLOC_MAX_WORKSPACE_BYTES)
// lives in every GPU that loads the library until the process exits.
#include <mutex>
#include <string>

#include "common.cuh"

namespace oasis {
cudaError_t launch_sparse_decode_attn(const Shape&, const uint16_t*, const uint16_t*, const uint16_t*,
                                      const int*, const int*, const int*, const int*, float, void*, float*,
                                      cudaStream_t);
size_t attn_workspace_bytes(const Shape&);
void set_last_error(const std::string&);
oasis_status validate_shape(const oasis_shape*, const char*, Shape*);
oasis_status validate_attn_args(const char*, const void*, const void*, const void*, const int32_t*, const int32_t*,
                                const int32_t*, const int32_t*, float, const float*);
}  // namespace oasis

namespace {

constexpr size_t kNoAllocWorkspaceBytes = OASIS_ATTN_NOALLOC_MAX_WORKSPACE_BYTES;
constexpr int kMaxDevices = 64;

// Shared by every call on a device; contents persist between calls.  The kernels
// write every partial they later read, so nothing has to start at zero.
static __device__ __align__(256) unsigned char g_attn_scratch[kNoAllocWorkspaceBytes];

std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_attn_scratch on the current device (looked up once per device).
cudaError_t scratch_for_current_device(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_attn_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

oasis_status fail(oasis_status st, const std::string& msg) {
  oasis::set_last_error("oasis_sparse_decode_attn_noalloc: " + msg);
  return st;
}

}  // namespace

extern "C" {

OASIS_API oasis_status oasis_sparse_decode_attn_noalloc(const oasis_shape* shape, const void* q, const void* k_pool,
                                                        const void* v_pool, const int32_t* sel, const int32_t* nsel,
                                                        const int32_t* blk2slot, const int32_t* ctx_len, float scale,
                                                        float* out, oasis_stream_t stream) {
  static const char* fn = "oasis_sparse_decode_attn_noalloc";
  // the same shape and argument checks (and messages) as oasis_sparse_decode_attn
  oasis::Shape s;
  oasis_status st = oasis::validate_shape(shape, fn, &s);
  if (st != OASIS_OK) return st;
  st = oasis::validate_attn_args(fn, q, k_pool, v_pool, sel, nsel, blk2slot, ctx_len, scale, out);
  if (st != OASIS_OK) return st;
  const size_t need = oasis::attn_workspace_bytes(s);
  if (need > kNoAllocWorkspaceBytes)
    return fail(OASIS_ERR_UNSUPPORTED, "this shape needs " + std::to_string(need) +
                                           " bytes of attention scratch, more than the built-in " +
                                           std::to_string(kNoAllocWorkspaceBytes) +
                                           " bytes; use oasis_sparse_decode_attn with a workspace");
  void* ws = nullptr;
  cudaError_t e = scratch_for_current_device(&ws);
  if (e == cudaSuccess)
    e = oasis::launch_sparse_decode_attn(s, static_cast<const uint16_t*>(q), static_cast<const uint16_t*>(k_pool),
                                         static_cast<const uint16_t*>(v_pool), sel, nsel, blk2slot, ctx_len, scale,
                                         ws, out, (cudaStream_t)stream);
  if (e != cudaSuccess)
    return fail(OASIS_ERR_CUDA, std::string(cudaGetErrorName(e)) + " (" + cudaGetErrorString(e) + ")");
  return OASIS_OK;
}

}  // extern "C"
