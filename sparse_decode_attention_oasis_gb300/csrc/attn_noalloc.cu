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

bool aligned_to(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

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
  if (!shape) return fail(OASIS_ERR_INVALID, "shape is NULL");
  const oasis_shape& sh = *shape;
  if (sh.B < 1 || sh.Hq < 1 || sh.Hkv < 1 || sh.nb_max < 1 || sh.n_la < 1 || sh.Kb < 1 || sh.P < 1 ||
      sh.Hq % sh.Hkv)
    return fail(OASIS_ERR_INVALID, "invalid shape");
  const int G = sh.Hq / sh.Hkv;
  if (sh.d != 128 || sh.bs != 16 || (G != 1 && G != 2 && G != 4 && G != 8) || sh.Kb > 256 || sh.P < sh.Kb ||
      sh.P > 1024 || sh.nb_max > 8192 || (long long)sh.B * sh.Hkv > 65535)
    return fail(OASIS_ERR_UNSUPPORTED, "shape outside the supported range");
  const oasis::Shape s{sh.B, sh.Hq, sh.Hkv, sh.d, sh.bs, sh.nb_max, sh.n_la, sh.Kb, sh.P};
  const size_t need = oasis::attn_workspace_bytes(s);
  if (need > kNoAllocWorkspaceBytes)
    return fail(OASIS_ERR_UNSUPPORTED, "this shape needs " + std::to_string(need) +
                                           " bytes of attention scratch, more than the built-in " +
                                           std::to_string(kNoAllocWorkspaceBytes) +
                                           " bytes; use oasis_sparse_decode_attn with a workspace");
  if (!q || !aligned_to(q, 16) || !k_pool || !v_pool || !aligned_to(k_pool, 16) || !aligned_to(v_pool, 16) ||
      !sel || !nsel || !blk2slot || !ctx_len || !out || !aligned_to(out, 16) || !aligned_to(sel, 4) ||
      !aligned_to(nsel, 4) || !aligned_to(blk2slot, 4) || !aligned_to(ctx_len, 4) || !(scale > 0.f))
    return fail(OASIS_ERR_INVALID, "bad pointer, alignment or scale");
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
