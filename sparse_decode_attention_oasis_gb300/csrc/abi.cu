// C ABI entry points: argument validation, then the kernel launches.
#include <atomic>
#include <mutex>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <string>

#include "fetch_copy.cuh"

namespace oasis {
cudaError_t launch_score_blocks(const Shape&, const uint16_t*, const int*, const uint16_t*, float2*, cudaStream_t);
cudaError_t launch_score_blocks_dyn(const Shape&, const uint16_t*, const int*, const uint16_t*, float2*, unsigned*, int,
                                    cudaStream_t);
bool score_tc_fits(const Shape& s);
cudaError_t launch_score_blocks_tc(const Shape&, const uint16_t*, const int*, const uint16_t*, float2*, unsigned*,
                                   cudaStream_t);
cudaError_t launch_topk_select(const Shape&, const float2*, const uint16_t*, const uint16_t*, const int*, int*,
                               int*, cudaStream_t);
cudaError_t launch_fetch_diff(const Shape&, const float2*, const uint16_t*, const uint16_t*, const int*,
                              const int*, const int*, const int*, int, int*, int*, cudaStream_t);
cudaError_t launch_gather_h2d(const Shape&, const uint16_t*, const int*, const int*, const int*, const int*,
                              int*, int*, int*, const int*, uint16_t*, uint16_t*, unsigned*, cudaStream_t);
cudaError_t launch_sparse_decode_attn(const Shape&, const uint16_t*, const uint16_t*, const uint16_t*,
                                      const int*, const int*, const int*, const int*, float, void*, float*,
                                      cudaStream_t);
size_t attn_workspace_bytes(const Shape&);
cudaError_t launch_assign_slots(const Shape&, const int*, const int*, const int*, const int*, int*, int*, int*,
                                const int*, unsigned*, cudaStream_t);
cudaError_t launch_copy_fetched(const Shape&, const CopyJob&, cudaStream_t);
cudaError_t launch_copy_fetched_wait(const Shape&, const CopyJob&, const unsigned*, unsigned, int, cudaStream_t);
cudaError_t launch_score_blocks_copy(const Shape&, const uint16_t*, const int*, const uint16_t*, float2*,
                                     const CopyJob&, cudaStream_t);
cudaError_t launch_set_agreement(const Shape&, const int*, const int*, const int*, const int*, const int*, int*,
                                 unsigned*, cudaStream_t);
cudaError_t launch_pool_keys(const Shape&, const uint16_t*, const int*, uint16_t*, cudaStream_t);
cudaError_t launch_pool_append(const Shape&, const uint16_t*, const int*, uint16_t*, unsigned*, cudaStream_t);
cudaError_t launch_score_pooled(const Shape&, const uint16_t*, const int*, const uint16_t*, float2*, const CopyJob*,
                                cudaStream_t);
cudaError_t launch_topk_select_pooled(const Shape&, const float2*, const uint16_t*, const uint16_t*, const int*,
                                      int*, int*, cudaStream_t);
cudaError_t launch_fetch_diff_pooled(const Shape&, const float2*, const uint16_t*, const uint16_t*, const int*,
                                     const int*, const int*, const int*, int, int*, int*, cudaStream_t);
cudaError_t launch_attn_lookahead(const Shape&, const uint16_t*, const uint16_t*, const uint16_t*, const uint16_t*,
                                  const int*, const int*, const int*, const int*, float, void*, float*, float*,
                                  cudaStream_t);
size_t attn_la_workspace_bytes(const Shape&);
cudaError_t launch_topk_select_diff(const Shape&, const float2*, const uint16_t*, const uint16_t*, const int*,
                                    const int*, int, int*, int*, int*, int*, bool, const uint16_t*, cudaStream_t);
cudaError_t launch_touch_host(const void*, size_t, unsigned*, cudaStream_t);
cudaError_t launch_append_kv(const Shape&, const uint16_t*, const uint16_t*, int*, uint16_t*, uint16_t*, const int*,
                             uint16_t*, uint16_t*, int, unsigned*, cudaStream_t);
size_t topk_smem_bytes(const Shape&);
}  // namespace oasis

namespace {

thread_local std::string g_last_error = "no error";

oasis_status fail(oasis_status st, const char* fn, const std::string& msg) {
  g_last_error = std::string(fn) + ": " + msg;
  return st;
}

oasis_status cuda_fail(const char* fn, cudaError_t e) {
  g_last_error = std::string(fn) + ": " + cudaGetErrorName(e) + " (" + cudaGetErrorString(e) + ")";
  return OASIS_ERR_CUDA;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Shape checks shared by every call.  Returns OK or the status to return.
oasis_status check_shape(const oasis_shape* sh, const char* fn, oasis::Shape* out) {
  if (!sh) return fail(OASIS_ERR_INVALID, fn, "shape is NULL");
  const oasis_shape& s = *sh;
  if (s.B < 1 || s.Hq < 1 || s.Hkv < 1 || s.nb_max < 1 || s.n_la < 1 || s.Kb < 1 || s.P < 1)
    return fail(OASIS_ERR_INVALID, fn, "every shape field must be >= 1");
  if (s.Hq % s.Hkv) return fail(OASIS_ERR_INVALID, fn, "Hq must be a multiple of Hkv");
  const int G = s.Hq / s.Hkv;
  if (s.d != 128) return fail(OASIS_ERR_UNSUPPORTED, fn, "head dim must be 128");
  if (s.bs != 16) return fail(OASIS_ERR_UNSUPPORTED, fn, "block size must be 16 tokens");
  if (G != 1 && G != 2 && G != 4 && G != 8) return fail(OASIS_ERR_UNSUPPORTED, fn, "GQA group must be 1, 2, 4 or 8");
  if (s.n_la * G > 32) return fail(OASIS_ERR_UNSUPPORTED, fn, "n_la * G must be <= 32");
  if (s.nb_max > 8192) return fail(OASIS_ERR_UNSUPPORTED, fn, "nb_max must be <= 8192");
  if (s.Kb > 256) return fail(OASIS_ERR_UNSUPPORTED, fn, "Kb must be <= 256");
  if (s.P < s.Kb || s.P > 1024) return fail(OASIS_ERR_UNSUPPORTED, fn, "P must be in [Kb, 1024]");
  if ((long long)s.B * s.Hkv > 65535) return fail(OASIS_ERR_UNSUPPORTED, fn, "B * Hkv must be <= 65535");
  *out = oasis::Shape{s.B, s.Hq, s.Hkv, s.d, s.bs, s.nb_max, s.n_la, s.Kb, s.P};
  return OASIS_OK;
}

}  // namespace

namespace {

#define REQUIRE(cond, msg) \
  do { if (!(cond)) return fail(OASIS_ERR_INVALID, fn, msg); } while (0)

}  // namespace

namespace oasis {
static std::mutex g_trace_mu;
static TraceBuf g_trace{nullptr, nullptr, 0};
TraceBuf trace_buf() {
  std::lock_guard<std::mutex> lk(g_trace_mu);
  return g_trace;
}
static std::atomic<int> g_score_ctas_per_sm{0};
static std::atomic<int> g_score_kernel{OASIS_SCORE_KERNEL_TC};  // tcgen05/TMA scorer unless set to mma.sync
static std::atomic<int> g_copy_ctas{0};     // 0: the copy kernel's own grid
int score_ctas_per_sm_option() { return g_score_ctas_per_sm.load(std::memory_order_relaxed); }
int copy_ctas_option() { return g_copy_ctas.load(std::memory_order_relaxed); }
static std::atomic<int> g_score_static_share{750};  // per mille, oasis_score_blocks_dynamic
int score_static_share_option() { return g_score_static_share.load(std::memory_order_relaxed); }
// Record the message oasis_last_error() returns on this thread.
void set_last_error(const std::string& msg) { g_last_error = msg; }

// The shape checks of every call, for entry points defined in other files.
oasis_status validate_shape(const oasis_shape* sh, const char* fn, Shape* out) { return check_shape(sh, fn, out); }

// The argument checks of the attention call other than its workspace (shared by
// oasis_sparse_decode_attn and its allocation-free variant, so the two accept
// and reject exactly the same arguments with the same messages).
oasis_status validate_attn_args(const char* fn, const void* q, const void* k_pool, const void* v_pool,
                                const int32_t* sel, const int32_t* nsel, const int32_t* blk2slot,
                                const int32_t* ctx_len, float scale, const float* out) {
  REQUIRE(q && aligned(q, 16), "q must be a 16-byte aligned device pointer");
  REQUIRE(k_pool && v_pool && aligned(k_pool, 16) && aligned(v_pool, 16),
          "k_pool/v_pool must be 16-byte aligned device pointers");
  REQUIRE(sel && nsel && blk2slot && ctx_len, "table pointers must be non-NULL");
  REQUIRE(aligned(sel, 4) && aligned(nsel, 4) && aligned(blk2slot, 4) && aligned(ctx_len, 4),
          "int32 arrays must be 4-byte aligned");
  REQUIRE(out && aligned(out, 16), "out must be a 16-byte aligned device pointer");
  REQUIRE(scale == scale && scale > 0.f, "scale must be a positive number");
  return OASIS_OK;
}
}  // namespace oasis

extern "C" {

const char* oasis_version(void) { return "oasis-gb300 0.1 sm_103a"; }

const char* oasis_last_error(void) { return g_last_error.c_str(); }

// Scoring kernel: TMA + tcgen05 (the default) or mma.sync from registers, chosen
// by oasis_set_option(OASIS_OPT_SCORE_KERNEL, ...); both implement the same
// definition and bound.  Shapes with more than 2^31 - 1 key rows in one layer
// (beyond the tensor map's 32-bit coordinates) take the mma.sync kernel.
static bool use_tc_scoring(const oasis::Shape& s) {
  return oasis::g_score_kernel.load(std::memory_order_relaxed) == OASIS_SCORE_KERNEL_TC && oasis::score_tc_fits(s);
}

// ------------------------------------------------------------------ span trace
static constexpr size_t kTraceHeaderBytes = 128;  // ctl words, padded

size_t oasis_trace_bytes(int32_t capacity) {
  if (capacity < 1) return 0;
  return kTraceHeaderBytes + (size_t)OASIS_TRACE_KINDS * (size_t)capacity * 2 * sizeof(unsigned long long);
}

oasis_status oasis_trace_set(void* dev_buf, int32_t capacity) {
  static const char* fn = "oasis_trace_set";
  if (dev_buf == nullptr) {
    std::lock_guard<std::mutex> lk(oasis::g_trace_mu);
    oasis::g_trace = oasis::TraceBuf{nullptr, nullptr, 0};
    return OASIS_OK;
  }
  REQUIRE(capacity >= 1, "capacity must be >= 1");
  REQUIRE(aligned(dev_buf, 16), "the trace buffer must be 16-byte aligned");
  std::lock_guard<std::mutex> lk(oasis::g_trace_mu);
  oasis::g_trace = oasis::TraceBuf{static_cast<unsigned*>(dev_buf),
                                   reinterpret_cast<unsigned long long*>(static_cast<char*>(dev_buf) + kTraceHeaderBytes),
                                   (int)capacity};
  return OASIS_OK;
}

oasis_status oasis_score_blocks(const oasis_shape* shape, const void* k_hbm, const int32_t* ctx_len,
                                const void* q_la, float* scores, uint32_t* err_word, oasis_stream_t stream) {
  static const char* fn = "oasis_score_blocks";
  oasis::Shape s;
  oasis_status st = check_shape(shape, fn, &s);
  if (st != OASIS_OK) return st;
  REQUIRE(k_hbm && aligned(k_hbm, 16), "k_hbm must be a 16-byte aligned device pointer");
  REQUIRE(q_la && aligned(q_la, 16), "q_la must be a 16-byte aligned device pointer");
  REQUIRE(ctx_len && aligned(ctx_len, 4), "ctx_len must be a 4-byte aligned device pointer");
  REQUIRE(scores && aligned(scores, 8), "scores must be an 8-byte aligned device pointer");
  REQUIRE(!err_word || aligned(err_word, 4), "err_word must be NULL or a 4-byte aligned device pointer");
  cudaError_t e = use_tc_scoring(s)
                      ? oasis::launch_score_blocks_tc(s, static_cast<const uint16_t*>(k_hbm), ctx_len,
                                                      static_cast<const uint16_t*>(q_la),
                                                      reinterpret_cast<float2*>(scores), err_word,
                                                      (cudaStream_t)stream)
                      : oasis::launch_score_blocks(s, static_cast<const uint16_t*>(k_hbm), ctx_len,
                                                   static_cast<const uint16_t*>(q_la),
                                                   reinterpret_cast<float2*>(scores), (cudaStream_t)stream);
  return e == cudaSuccess ? OASIS_OK : cuda_fail(fn, e);
}

oasis_status oasis_score_blocks_dynamic(const oasis_shape* shape, const void* k_hbm, const int32_t* ctx_len,
                                        const void* q_la, float* scores, uint32_t* work, int32_t reserve_ctas,
                                        oasis_stream_t stream) {
  static const char* fn = "oasis_score_blocks_dynamic";
  oasis::Shape s;
  oasis_status st = check_shape(shape, fn, &s);
  if (st != OASIS_OK) return st;
  REQUIRE(k_hbm && aligned(k_hbm, 16), "k_hbm must be a 16-byte aligned device pointer");
  REQUIRE(q_la && aligned(q_la, 16), "q_la must be a 16-byte aligned device pointer");
  REQUIRE(ctx_len && aligned(ctx_len, 4), "ctx_len must be a 4-byte aligned device pointer");
  REQUIRE(scores && aligned(scores, 8), "scores must be an 8-byte aligned device pointer");
  REQUIRE(work && aligned(work, 8), "work must be an 8-byte aligned device pointer to two uint32");
  REQUIRE(reserve_ctas >= 0 && reserve_ctas <= 4096, "reserve_ctas must be in [0, 4096]");
  cudaError_t e = oasis::launch_score_blocks_dyn(s, static_cast<const uint16_t*>(k_hbm), ctx_len,
                                                 static_cast<const uint16_t*>(q_la), reinterpret_cast<float2*>(scores),
                                                 work, reserve_ctas, (cudaStream_t)stream);
  return e == cudaSuccess ? OASIS_OK : cuda_fail(fn, e);
}

oasis_status oasis_topk_select(const oasis_shape* shape, const float* scores, const void* k_hbm,
                               const void* q_la, const int32_t* ctx_len, int32_t* sel, int32_t* nsel,
                               oasis_stream_t stream) {
  static const char* fn = "oasis_topk_select";
  oasis::Shape s;
  oasis_status st = check_shape(shape, fn, &s);
  if (st != OASIS_OK) return st;
  REQUIRE(scores && aligned(scores, 8), "scores must be an 8-byte aligned device pointer");
  REQUIRE(k_hbm && aligned(k_hbm, 16), "k_hbm must be a 16-byte aligned device pointer");
  REQUIRE(q_la && aligned(q_la, 16), "q_la must be a 16-byte aligned device pointer");
  REQUIRE(ctx_len && aligned(ctx_len, 4), "ctx_len must be a 4-byte aligned device pointer");
  REQUIRE(sel && aligned(sel, 4) && nsel && aligned(nsel, 4), "sel/nsel must be 4-byte aligned device pointers");
  cudaError_t e = oasis::launch_topk_select(s, reinterpret_cast<const float2*>(scores),
                                            static_cast<const uint16_t*>(k_hbm),
                                            static_cast<const uint16_t*>(q_la), ctx_len, sel, nsel,
                                            (cudaStream_t)stream);
  return e == cudaSuccess ? OASIS_OK : cuda_fail(fn, e);
}

oasis_status oasis_fetch_diff_capped(const oasis_shape* shape, const float* scores, const void* k_hbm,
                                     const void* q_la, const int32_t* ctx_len, const int32_t* sel,
                                     const int32_t* nsel, const int32_t* blk2slot, int32_t fetch_cap,
                                     int32_t* fetch, int32_t* nfetch, oasis_stream_t stream) {
  static const char* fn = "oasis_fetch_diff_capped";
  oasis::Shape s;
  oasis_status st = check_shape(shape, fn, &s);
  if (st != OASIS_OK) return st;
  REQUIRE(scores && aligned(scores, 8), "scores must be an 8-byte aligned device pointer");
  REQUIRE(k_hbm && aligned(k_hbm, 16), "k_hbm must be a 16-byte aligned device pointer");
  REQUIRE(q_la && aligned(q_la, 16), "q_la must be a 16-byte aligned device pointer");
  REQUIRE(ctx_len && aligned(ctx_len, 4), "ctx_len must be a 4-byte aligned device pointer");
  REQUIRE(sel && nsel && blk2slot && fetch && nfetch, "sel/nsel/blk2slot/fetch/nfetch must be device pointers");
  REQUIRE(aligned(sel, 4) && aligned(nsel, 4) && aligned(blk2slot, 4) && aligned(fetch, 4) && aligned(nfetch, 4),
          "int32 arrays must be 4-byte aligned");
  REQUIRE(fetch_cap >= 0 && fetch_cap <= s.Kb, "fetch_cap must be in [0, Kb]");
  cudaError_t e = oasis::launch_fetch_diff(s, reinterpret_cast<const float2*>(scores),
                                           static_cast<const uint16_t*>(k_hbm),
                                           static_cast<const uint16_t*>(q_la), ctx_len, sel, nsel, blk2slot,
                                           fetch_cap, fetch, nfetch, (cudaStream_t)stream);
  return e == cudaSuccess ? OASIS_OK : cuda_fail(fn, e);
}

// Device address of page-locked mapped host memory (NULL if `p` is not such memory).
static void* mapped_host_ptr(const void* p) {
  cudaPointerAttributes attr;
  if (cudaPointerGetAttributes(&attr, p) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  if (attr.type != cudaMemoryTypeHost) return nullptr;
  return attr.devicePointer;
}

oasis_status oasis_gather_h2d(const oasis_shape* shape, const void* host_kv, const int32_t* sel,
                              const int32_t* nsel, const int32_t* fetch, const int32_t* nfetch,
                              int32_t* blk2slot, int32_t* slot2blk, int32_t* last_used, const int32_t* step,
                              void* k_pool, void* v_pool, uint32_t* err_word, oasis_stream_t stream) {
  static const char* fn = "oasis_gather_h2d";
  oasis::Shape s;
  oasis_status st = check_shape(shape, fn, &s);
  if (st != OASIS_OK) return st;
  REQUIRE(host_kv && aligned(host_kv, 16), "host_kv must be a 16-byte aligned pointer");
  REQUIRE(k_pool && v_pool && aligned(k_pool, 16) && aligned(v_pool, 16),
          "k_pool/v_pool must be 16-byte aligned device pointers");
  REQUIRE(sel && nsel && fetch && nfetch && blk2slot && slot2blk && last_used && err_word && step,
          "table pointers must be non-NULL");
  REQUIRE(aligned(step, 4), "step must be a 4-byte aligned device pointer");
  REQUIRE(aligned(sel, 4) && aligned(nsel, 4) && aligned(fetch, 4) && aligned(nfetch, 4) &&
              aligned(blk2slot, 4) && aligned(slot2blk, 4) && aligned(last_used, 4) && aligned(err_word, 4),
          "int32 arrays must be 4-byte aligned");
  // The host tier must be page-locked host memory mapped into the device address space.
  cudaPointerAttributes attr;
  cudaError_t e = cudaPointerGetAttributes(&attr, host_kv);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(OASIS_ERR_INVALID, fn, "host_kv is not a CUDA-registered pointer");
  }
  if (attr.type != cudaMemoryTypeHost || attr.devicePointer == nullptr)
    return fail(OASIS_ERR_INVALID, fn, "host_kv must be page-locked, device-mapped host memory");
  e = oasis::launch_gather_h2d(s, static_cast<const uint16_t*>(attr.devicePointer), sel, nsel, fetch, nfetch,
                               blk2slot, slot2blk, last_used, step, static_cast<uint16_t*>(k_pool),
                               static_cast<uint16_t*>(v_pool), err_word, (cudaStream_t)stream);
  return e == cudaSuccess ? OASIS_OK : cuda_fail(fn, e);
}


oasis_status oasis_assign_slots(const oasis_shape* shape, const int32_t* sel, const int32_t* nsel,
                                const int32_t* fetch, const int32_t* nfetch, int32_t* blk2slot,
                                int32_t* slot2blk, int32_t* last_used, const int32_t* step, uint32_t* err_word,
                                oasis_stream_t stream) {
  static const char* fn = "oasis_assign_slots";
  oasis::Shape s;
  oasis_status st = check_shape(shape, fn, &s);
  if (st != OASIS_OK) return st;
  REQUIRE(sel && nsel && fetch && nfetch && blk2slot && slot2blk && last_used && err_word && step,
          "table pointers must be non-NULL");
  REQUIRE(aligned(sel, 4) && aligned(nsel, 4) && aligned(fetch, 4) && aligned(nfetch, 4) &&
              aligned(blk2slot, 4) && aligned(slot2blk, 4) && aligned(last_used, 4) && aligned(err_word, 4) &&
              aligned(step, 4),
          "int32 arrays must be 4-byte aligned");
  cudaError_t e = oasis::launch_assign_slots(s, sel, nsel, fetch, nfetch, blk2slot, slot2blk, last_used, step,
                                             err_word, (cudaStream_t)stream);
  return e == cudaSuccess ? OASIS_OK : cuda_fail(fn, e);
}

// Validate the copy arguments and build the job (device address of the host tier).
static oasis_status make_copy_job(const char* fn, const void* host_kv, const int32_t* fetch,
                                  const int32_t* nfetch, const int32_t* blk2slot, void* k_pool, void* v_pool,
                                  uint32_t* err_word, oasis::CopyJob* job) {
  REQUIRE(host_kv && aligned(host_kv, 16), "host_kv must be a 16-byte aligned pointer");
  REQUIRE(k_pool && v_pool && aligned(k_pool, 16) && aligned(v_pool, 16),
          "k_pool/v_pool must be 16-byte aligned device pointers");
  REQUIRE(fetch && nfetch && blk2slot && err_word, "fetch, nfetch, blk2slot and err_word must be non-NULL");
  REQUIRE(aligned(fetch, 4) && aligned(nfetch, 4) && aligned(blk2slot, 4) && aligned(err_word, 4),
          "int32 arrays must be 4-byte aligned");
  void* dev_host = mapped_host_ptr(host_kv);
  REQUIRE(dev_host, "host_kv must be page-locked, device-mapped host memory");
  *job = oasis::CopyJob{static_cast<const uint16_t*>(dev_host), fetch, nfetch, blk2slot,
                        static_cast<uint16_t*>(k_pool), static_cast<uint16_t*>(v_pool), err_word};
  return OASIS_OK;
}

oasis_status oasis_copy_fetched(const oasis_shape* shape, const void* host_kv, const int32_t* fetch,
                                const int32_t* nfetch, const int32_t* blk2slot, void* k_pool, void* v_pool,
                                uint32_t* err_word, oasis_stream_t stream) {
  static const char* fn = "oasis_copy_fetched";
  oasis::Shape s;
  oasis_status st = check_shape(shape, fn, &s);
  if (st != OASIS_OK) return st;
  oasis::CopyJob job;
  st = make_copy_job(fn, host_kv, fetch, nfetch, blk2slot, k_pool, v_pool, err_word, &job);
  if (st != OASIS_OK) return st;
  cudaError_t e = oasis::launch_copy_fetched(s, job, (cudaStream_t)stream);
  return e == cudaSuccess ? OASIS_OK : cuda_fail(fn, e);
}

oasis_status oasis_copy_fetched_wait(const oasis_shape* shape, const void* host_kv, const int32_t* fetch,
                                     const int32_t* nfetch, const int32_t* blk2slot, void* k_pool, void* v_pool,
                                     const uint32_t* ready_flag, uint32_t ready_value, int32_t max_polls,
                                     uint32_t* err_word, oasis_stream_t stream) {
  static const char* fn = "oasis_copy_fetched_wait";
  oasis::Shape s;
  oasis_status st = check_shape(shape, fn, &s);
  if (st != OASIS_OK) return st;
  oasis::CopyJob job;
  st = make_copy_job(fn, host_kv, fetch, nfetch, blk2slot, k_pool, v_pool, err_word, &job);
  if (st != OASIS_OK) return st;
  REQUIRE(ready_flag && aligned(ready_flag, 4), "ready_flag must be a 4-byte aligned pointer");
  REQUIRE(max_polls >= 1 && max_polls <= OASIS_MAX_READY_POLLS, "max_polls must be in [1, OASIS_MAX_READY_POLLS]");
  void* dev_flag = mapped_host_ptr(ready_flag);
  REQUIRE(dev_flag, "ready_flag must be in page-locked, device-mapped host memory");
  cudaError_t e = oasis::launch_copy_fetched_wait(s, job, static_cast<const unsigned*>(dev_flag), ready_value,
                                                  max_polls, (cudaStream_t)stream);
  return e == cudaSuccess ? OASIS_OK : cuda_fail(fn, e);
}

oasis_status oasis_error_word_status(const uint32_t* err_word, oasis_stream_t stream, uint32_t* bits) {
  static const char* fn = "oasis_error_word_status";
  REQUIRE(err_word && aligned(err_word, 4), "err_word must be a 4-byte aligned device pointer");
  cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(fn, e);
  uint32_t v = 0;
  e = cudaMemcpy(&v, err_word, sizeof(v), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(fn, e);
  if (bits) *bits = v;
  if (v & OASIS_EW_TIMEOUT) return fail(OASIS_ERR_TIMEOUT, fn, "a bounded wait on a host flag gave up");
  return OASIS_OK;
}

oasis_status oasis_score_blocks_copy(const oasis_shape* shape, const void* k_hbm, const int32_t* ctx_len,
                                     const void* q_la, float* scores, const void* host_kv, const int32_t* fetch,
                                     const int32_t* nfetch, const int32_t* blk2slot, void* k_pool, void* v_pool,
                                     uint32_t* err_word, oasis_stream_t stream) {
  static const char* fn = "oasis_score_blocks_copy";
  oasis::Shape s;
  oasis_status st = check_shape(shape, fn, &s);
  if (st != OASIS_OK) return st;
  REQUIRE(k_hbm && aligned(k_hbm, 16), "k_hbm must be a 16-byte aligned device pointer");
  REQUIRE(q_la && aligned(q_la, 16), "q_la must be a 16-byte aligned device pointer");
  REQUIRE(ctx_len && aligned(ctx_len, 4), "ctx_len must be a 4-byte aligned device pointer");
  REQUIRE(scores && aligned(scores, 8), "scores must be an 8-byte aligned device pointer");
  oasis::CopyJob job;
  st = make_copy_job(fn, host_kv, fetch, nfetch, blk2slot, k_pool, v_pool, err_word, &job);
  if (st != OASIS_OK) return st;
  const auto* k = static_cast<const uint16_t*>(k_hbm);
  const auto* q = static_cast<const uint16_t*>(q_la);
  auto* sc = reinterpret_cast<float2*>(scores);
  cudaError_t e;
  if (use_tc_scoring(s)) {
    e = oasis::launch_score_blocks_tc(s, k, ctx_len, q, sc, err_word, (cudaStream_t)stream);
    if (e == cudaSuccess) e = oasis::launch_copy_fetched(s, job, (cudaStream_t)stream);
  } else {
    e = oasis::launch_score_blocks_copy(s, k, ctx_len, q, sc, job, (cudaStream_t)stream);
  }
  return e == cudaSuccess ? OASIS_OK : cuda_fail(fn, e);
}

oasis_status oasis_pool_keys(const oasis_shape* shape, const void* k_hbm, const int32_t* ctx_len, void* k_pooled,
                             oasis_stream_t stream) {
  static const char* fn = "oasis_pool_keys";
  oasis::Shape s;
  oasis_status st = check_shape(shape, fn, &s);
  if (st != OASIS_OK) return st;
  REQUIRE(k_hbm && aligned(k_hbm, 16), "k_hbm must be a 16-byte aligned device pointer");
  REQUIRE(k_pooled && aligned(k_pooled, 16), "k_pooled must be a 16-byte aligned device pointer");
  REQUIRE(ctx_len && aligned(ctx_len, 4), "ctx_len must be a 4-byte aligned device pointer");
  cudaError_t e = oasis::launch_pool_keys(s, static_cast<const uint16_t*>(k_hbm), ctx_len,
                                          static_cast<uint16_t*>(k_pooled), (cudaStream_t)stream);
  return e == cudaSuccess ? OASIS_OK : cuda_fail(fn, e);
}

oasis_status oasis_pool_append(const oasis_shape* shape, const void* k_new, const int32_t* ctx_len, void* k_pooled,
                               uint32_t* err_word, oasis_stream_t stream) {
  static const char* fn = "oasis_pool_append";
  oasis::Shape s;
  oasis_status st = check_shape(shape, fn, &s);
  if (st != OASIS_OK) return st;
  REQUIRE(k_new && aligned(k_new, 16), "k_new must be a 16-byte aligned device pointer");
  REQUIRE(k_pooled && aligned(k_pooled, 16), "k_pooled must be a 16-byte aligned device pointer");
  REQUIRE(ctx_len && aligned(ctx_len, 4), "ctx_len must be a 4-byte aligned device pointer");
  REQUIRE(!err_word || aligned(err_word, 4), "err_word must be NULL or 4-byte aligned");
  cudaError_t e = oasis::launch_pool_append(s, static_cast<const uint16_t*>(k_new), ctx_len,
                                            static_cast<uint16_t*>(k_pooled), err_word, (cudaStream_t)stream);
  return e == cudaSuccess ? OASIS_OK : cuda_fail(fn, e);
}

oasis_status oasis_score_blocks_pooled(const oasis_shape* shape, const void* k_pooled, const int32_t* ctx_len,
                                       const void* q_la, float* scores, const void* host_kv, const int32_t* fetch,
                                       const int32_t* nfetch, const int32_t* blk2slot, void* k_pool,
                                       void* v_pool, uint32_t* err_word, oasis_stream_t stream) {
  static const char* fn = "oasis_score_blocks_pooled";
  oasis::Shape s;
  oasis_status st = check_shape(shape, fn, &s);
  if (st != OASIS_OK) return st;
  REQUIRE(k_pooled && aligned(k_pooled, 16), "k_pooled must be a 16-byte aligned device pointer");
  REQUIRE(q_la && aligned(q_la, 16), "q_la must be a 16-byte aligned device pointer");
  REQUIRE(ctx_len && aligned(ctx_len, 4), "ctx_len must be a 4-byte aligned device pointer");
  REQUIRE(scores && aligned(scores, 8), "scores must be an 8-byte aligned device pointer");
  oasis::CopyJob job;
  const bool copy = host_kv != nullptr;
  if (copy) {
    st = make_copy_job(fn, host_kv, fetch, nfetch, blk2slot, k_pool, v_pool, err_word, &job);
    if (st != OASIS_OK) return st;
  }
  cudaError_t e = oasis::launch_score_pooled(s, static_cast<const uint16_t*>(k_pooled), ctx_len,
                                             static_cast<const uint16_t*>(q_la), reinterpret_cast<float2*>(scores),
                                             copy ? &job : nullptr, (cudaStream_t)stream);
  return e == cudaSuccess ? OASIS_OK : cuda_fail(fn, e);
}

oasis_status oasis_topk_select_pooled(const oasis_shape* shape, const float* scores, const void* k_pooled,
                                      const void* q_la, const int32_t* ctx_len, int32_t* sel, int32_t* nsel,
                                      oasis_stream_t stream) {
  static const char* fn = "oasis_topk_select_pooled";
  oasis::Shape s;
  oasis_status st = check_shape(shape, fn, &s);
  if (st != OASIS_OK) return st;
  REQUIRE(scores && aligned(scores, 8), "scores must be an 8-byte aligned device pointer");
  REQUIRE(k_pooled && aligned(k_pooled, 16), "k_pooled must be a 16-byte aligned device pointer");
  REQUIRE(q_la && aligned(q_la, 16), "q_la must be a 16-byte aligned device pointer");
  REQUIRE(ctx_len && aligned(ctx_len, 4), "ctx_len must be a 4-byte aligned device pointer");
  REQUIRE(sel && aligned(sel, 4) && nsel && aligned(nsel, 4), "sel/nsel must be 4-byte aligned device pointers");
  cudaError_t e = oasis::launch_topk_select_pooled(s, reinterpret_cast<const float2*>(scores),
                                                   static_cast<const uint16_t*>(k_pooled),
                                                   static_cast<const uint16_t*>(q_la), ctx_len, sel, nsel,
                                                   (cudaStream_t)stream);
  return e == cudaSuccess ? OASIS_OK : cuda_fail(fn, e);
}

oasis_status oasis_fetch_diff_capped_pooled(const oasis_shape* shape, const float* scores, const void* k_pooled,
                                            const void* q_la, const int32_t* ctx_len, const int32_t* sel,
                                            const int32_t* nsel, const int32_t* blk2slot, int32_t fetch_cap,
                                            int32_t* fetch, int32_t* nfetch, oasis_stream_t stream) {
  static const char* fn = "oasis_fetch_diff_capped_pooled";
  oasis::Shape s;
  oasis_status st = check_shape(shape, fn, &s);
  if (st != OASIS_OK) return st;
  REQUIRE(scores && aligned(scores, 8), "scores must be an 8-byte aligned device pointer");
  REQUIRE(k_pooled && aligned(k_pooled, 16), "k_pooled must be a 16-byte aligned device pointer");
  REQUIRE(q_la && aligned(q_la, 16), "q_la must be a 16-byte aligned device pointer");
  REQUIRE(ctx_len && aligned(ctx_len, 4), "ctx_len must be a 4-byte aligned device pointer");
  REQUIRE(sel && nsel && blk2slot && fetch && nfetch, "sel/nsel/blk2slot/fetch/nfetch must be device pointers");
  REQUIRE(aligned(sel, 4) && aligned(nsel, 4) && aligned(blk2slot, 4) && aligned(fetch, 4) && aligned(nfetch, 4),
          "int32 arrays must be 4-byte aligned");
  REQUIRE(fetch_cap >= 0 && fetch_cap <= s.Kb, "fetch_cap must be in [0, Kb]");
  cudaError_t e = oasis::launch_fetch_diff_pooled(s, reinterpret_cast<const float2*>(scores),
                                                  static_cast<const uint16_t*>(k_pooled),
                                                  static_cast<const uint16_t*>(q_la), ctx_len, sel, nsel, blk2slot,
                                                  fetch_cap, fetch, nfetch, (cudaStream_t)stream);
  return e == cudaSuccess ? OASIS_OK : cuda_fail(fn, e);
}

size_t oasis_attn_lookahead_workspace_bytes(const oasis_shape* shape) {
  oasis::Shape s;
  if (check_shape(shape, "oasis_attn_lookahead_workspace_bytes", &s) != OASIS_OK) return 0;
  return oasis::attn_la_workspace_bytes(s);
}

oasis_status oasis_sparse_decode_attn_lookahead(const oasis_shape* shape, const void* q, const void* q_la,
                                                const void* k_pool, const void* v_pool, const int32_t* sel,
                                                const int32_t* nsel, const int32_t* blk2slot,
                                                const int32_t* ctx_len, float scale, void* workspace,
                                                size_t ws_bytes, float* out, float* out_la,
                                                oasis_stream_t stream) {
  static const char* fn = "oasis_sparse_decode_attn_lookahead";
  oasis::Shape s;
  oasis_status st = check_shape(shape, fn, &s);
  if (st != OASIS_OK) return st;
  REQUIRE(q && aligned(q, 16) && q_la && aligned(q_la, 16), "q and q_la must be 16-byte aligned device pointers");
  REQUIRE(k_pool && v_pool && aligned(k_pool, 16) && aligned(v_pool, 16),
          "k_pool/v_pool must be 16-byte aligned device pointers");
  REQUIRE(sel && nsel && blk2slot && ctx_len, "table pointers must be non-NULL");
  REQUIRE(aligned(sel, 4) && aligned(nsel, 4) && aligned(blk2slot, 4) && aligned(ctx_len, 4),
          "int32 arrays must be 4-byte aligned");
  REQUIRE(out && aligned(out, 16) && out_la && aligned(out_la, 16),
          "out and out_la must be 16-byte aligned device pointers");
  REQUIRE(workspace && aligned(workspace, 16), "workspace must be a 16-byte aligned device pointer");
  REQUIRE(ws_bytes >= oasis::attn_la_workspace_bytes(s),
          "workspace is smaller than oasis_attn_lookahead_workspace_bytes()");
  REQUIRE(scale == scale && scale > 0.f, "scale must be a positive number");
  cudaError_t e = oasis::launch_attn_lookahead(s, static_cast<const uint16_t*>(q), static_cast<const uint16_t*>(q_la),
                                               static_cast<const uint16_t*>(k_pool),
                                               static_cast<const uint16_t*>(v_pool), sel, nsel, blk2slot, ctx_len,
                                               scale, workspace, out, out_la, (cudaStream_t)stream);
  return e == cudaSuccess ? OASIS_OK : cuda_fail(fn, e);
}

static oasis_status topk_diff_call(const char* fn, const oasis_shape* shape, const float* scores, const void* keys,
                                   const void* q_la, const int32_t* ctx_len, const int32_t* blk2slot,
                                   int32_t fetch_cap, int32_t* sel, int32_t* nsel, int32_t* fetch, int32_t* nfetch,
                                   const void* host_kv, bool pooled, oasis_stream_t stream) {
  oasis::Shape s;
  oasis_status st = check_shape(shape, fn, &s);
  if (st != OASIS_OK) return st;
  REQUIRE(scores && aligned(scores, 8), "scores must be an 8-byte aligned device pointer");
  REQUIRE(keys && aligned(keys, 16), "the key pointer must be a 16-byte aligned device pointer");
  REQUIRE(q_la && aligned(q_la, 16), "q_la must be a 16-byte aligned device pointer");
  REQUIRE(ctx_len && aligned(ctx_len, 4), "ctx_len must be a 4-byte aligned device pointer");
  REQUIRE(sel && nsel && blk2slot && fetch && nfetch, "sel/nsel/blk2slot/fetch/nfetch must be device pointers");
  REQUIRE(aligned(sel, 4) && aligned(nsel, 4) && aligned(blk2slot, 4) && aligned(fetch, 4) && aligned(nfetch, 4),
          "int32 arrays must be 4-byte aligned");
  REQUIRE(fetch_cap >= 0 && fetch_cap <= s.Kb, "fetch_cap must be in [0, Kb]");
  const void* dev_host = nullptr;
  if (host_kv) {
    REQUIRE(aligned(host_kv, 16), "host_kv must be 16-byte aligned");
    dev_host = mapped_host_ptr(host_kv);
    REQUIRE(dev_host, "host_kv must be page-locked, device-mapped host memory");
  }
  cudaError_t e = oasis::launch_topk_select_diff(s, reinterpret_cast<const float2*>(scores),
                                                 static_cast<const uint16_t*>(keys),
                                                 static_cast<const uint16_t*>(q_la), ctx_len, blk2slot, fetch_cap,
                                                 sel, nsel, fetch, nfetch, pooled,
                                                 static_cast<const uint16_t*>(dev_host), (cudaStream_t)stream);
  return e == cudaSuccess ? OASIS_OK : cuda_fail(fn, e);
}

oasis_status oasis_topk_select_diff(const oasis_shape* shape, const float* scores, const void* k_hbm,
                                    const void* q_la, const int32_t* ctx_len, const int32_t* blk2slot,
                                    int32_t fetch_cap, int32_t* sel, int32_t* nsel, int32_t* fetch,
                                    int32_t* nfetch, const void* host_kv, oasis_stream_t stream) {
  return topk_diff_call("oasis_topk_select_diff", shape, scores, k_hbm, q_la, ctx_len, blk2slot, fetch_cap, sel,
                        nsel, fetch, nfetch, host_kv, false, stream);
}

oasis_status oasis_topk_select_diff_pooled(const oasis_shape* shape, const float* scores, const void* k_pooled,
                                           const void* q_la, const int32_t* ctx_len, const int32_t* blk2slot,
                                           int32_t fetch_cap, int32_t* sel, int32_t* nsel, int32_t* fetch,
                                           int32_t* nfetch, const void* host_kv, oasis_stream_t stream) {
  return topk_diff_call("oasis_topk_select_diff_pooled", shape, scores, k_pooled, q_la, ctx_len, blk2slot,
                        fetch_cap, sel, nsel, fetch, nfetch, host_kv, true, stream);
}

oasis_status oasis_set_option(int32_t option, int32_t value) {
  static const char* fn = "oasis_set_option";
  if (option == OASIS_OPT_SCORE_CTAS_PER_SM) {
    REQUIRE(value >= 0 && value <= 64, "OASIS_OPT_SCORE_CTAS_PER_SM takes 0 (the kernel's choice) to 64");
    oasis::g_score_ctas_per_sm.store(value, std::memory_order_relaxed);
    return OASIS_OK;
  }
  if (option == OASIS_OPT_COPY_CTAS) {
    REQUIRE(value >= 0 && value <= 65535, "OASIS_OPT_COPY_CTAS takes 0 (the kernel's choice) to 65535");
    oasis::g_copy_ctas.store(value, std::memory_order_relaxed);
    return OASIS_OK;
  }
  if (option == OASIS_OPT_SCORE_STATIC_SHARE) {
    REQUIRE(value >= 0 && value <= 1000, "OASIS_OPT_SCORE_STATIC_SHARE takes 0 to 1000 (per mille)");
    oasis::g_score_static_share.store(value, std::memory_order_relaxed);
    return OASIS_OK;
  }
  if (option == OASIS_OPT_SCORE_KERNEL) {
    REQUIRE(value == OASIS_SCORE_KERNEL_MMA || value == OASIS_SCORE_KERNEL_TC,
            "OASIS_OPT_SCORE_KERNEL takes OASIS_SCORE_KERNEL_MMA or OASIS_SCORE_KERNEL_TC");
    oasis::g_score_kernel.store(value, std::memory_order_relaxed);
    return OASIS_OK;
  }
  return fail(OASIS_ERR_INVALID, fn, "unknown option");
}

oasis_status oasis_set_agreement(const oasis_shape* shape, const int32_t* pred, const int32_t* npred,
                                 const int32_t* exact, const int32_t* nexact, const int32_t* blk2slot,
                                 int32_t* counts, uint32_t* err_word, oasis_stream_t stream) {
  static const char* fn = "oasis_set_agreement";
  oasis::Shape s;
  oasis_status st = check_shape(shape, fn, &s);
  if (st != OASIS_OK) return st;
  REQUIRE(pred && npred && exact && nexact && counts, "pred, npred, exact, nexact and counts must be non-NULL");
  REQUIRE(aligned(pred, 4) && aligned(npred, 4) && aligned(exact, 4) && aligned(nexact, 4) && aligned(counts, 4) &&
              (!blk2slot || aligned(blk2slot, 4)) && (!err_word || aligned(err_word, 4)),
          "int32 arrays must be 4-byte aligned");
  cudaError_t e = oasis::launch_set_agreement(s, pred, npred, exact, nexact, blk2slot, counts, err_word,
                                              (cudaStream_t)stream);
  return e == cudaSuccess ? OASIS_OK : cuda_fail(fn, e);
}

oasis_status oasis_touch_host(const void* host_ptr, size_t bytes, uint32_t* sink, oasis_stream_t stream) {
  static const char* fn = "oasis_touch_host";
  REQUIRE(host_ptr && aligned(host_ptr, 16), "host_ptr must be a 16-byte aligned pointer");
  REQUIRE(bytes % 16 == 0, "bytes must be a multiple of 16");
  REQUIRE(!sink || aligned(sink, 4), "sink must be NULL or a 4-byte aligned device pointer");
  void* dev = mapped_host_ptr(host_ptr);
  REQUIRE(dev, "host_ptr must be page-locked, device-mapped host memory");
  cudaError_t e = oasis::launch_touch_host(dev, bytes, sink, (cudaStream_t)stream);
  return e == cudaSuccess ? OASIS_OK : cuda_fail(fn, e);
}

oasis_status oasis_append_kv(const oasis_shape* shape, const void* k_new, const void* v_new, int32_t* ctx_len,
                             void* k_hbm, void* host_kv, const int32_t* blk2slot, void* k_pool, void* v_pool,
                             int32_t advance, uint32_t* err_word, oasis_stream_t stream) {
  static const char* fn = "oasis_append_kv";
  oasis::Shape s;
  oasis_status st = check_shape(shape, fn, &s);
  if (st != OASIS_OK) return st;
  REQUIRE(k_new && v_new && aligned(k_new, 16) && aligned(v_new, 16), "k_new/v_new must be 16-byte aligned");
  REQUIRE(k_hbm && aligned(k_hbm, 16), "k_hbm must be a 16-byte aligned device pointer");
  REQUIRE(k_pool && v_pool && aligned(k_pool, 16) && aligned(v_pool, 16), "pools must be 16-byte aligned");
  REQUIRE(ctx_len && aligned(ctx_len, 4) && blk2slot && aligned(blk2slot, 4), "ctx_len/blk2slot must be int32 arrays");
  REQUIRE(!err_word || aligned(err_word, 4), "err_word must be NULL or 4-byte aligned");
  REQUIRE(host_kv && aligned(host_kv, 16), "host_kv must be a 16-byte aligned pointer");
  void* host_dev = mapped_host_ptr(host_kv);
  if (!host_dev) return fail(OASIS_ERR_INVALID, fn, "host_kv must be page-locked, device-mapped host memory");
  cudaError_t e = oasis::launch_append_kv(s, static_cast<const uint16_t*>(k_new), static_cast<const uint16_t*>(v_new),
                                          ctx_len, static_cast<uint16_t*>(k_hbm), static_cast<uint16_t*>(host_dev),
                                          blk2slot, static_cast<uint16_t*>(k_pool), static_cast<uint16_t*>(v_pool),
                                          advance, err_word, (cudaStream_t)stream);
  return e == cudaSuccess ? OASIS_OK : cuda_fail(fn, e);
}

size_t oasis_attn_workspace_bytes(const oasis_shape* shape) {
  oasis::Shape s;
  if (check_shape(shape, "oasis_attn_workspace_bytes", &s) != OASIS_OK) return 0;
  return oasis::attn_workspace_bytes(s);
}

oasis_status oasis_sparse_decode_attn(const oasis_shape* shape, const void* q, const void* k_pool,
                                      const void* v_pool, const int32_t* sel, const int32_t* nsel,
                                      const int32_t* blk2slot, const int32_t* ctx_len, float scale,
                                      void* workspace, size_t ws_bytes, float* out, oasis_stream_t stream) {
  static const char* fn = "oasis_sparse_decode_attn";
  oasis::Shape s;
  oasis_status st = check_shape(shape, fn, &s);
  if (st != OASIS_OK) return st;
  st = oasis::validate_attn_args(fn, q, k_pool, v_pool, sel, nsel, blk2slot, ctx_len, scale, out);
  if (st != OASIS_OK) return st;
  REQUIRE(workspace && aligned(workspace, 16), "workspace must be a 16-byte aligned device pointer");
  REQUIRE(ws_bytes >= oasis::attn_workspace_bytes(s), "workspace is smaller than oasis_attn_workspace_bytes()");
  cudaError_t e = oasis::launch_sparse_decode_attn(s, static_cast<const uint16_t*>(q),
                                                   static_cast<const uint16_t*>(k_pool),
                                                   static_cast<const uint16_t*>(v_pool), sel, nsel, blk2slot,
                                                   ctx_len, scale, workspace, out, (cudaStream_t)stream);
  return e == cudaSuccess ? OASIS_OK : cuda_fail(fn, e);
}

}  // extern "C"
