/*
 * oasis.h - C ABI of the GB300 (sm_103a) lookahead sparse decode hot path.
 *
 * The method (OasisKV: Scaling In-Decode KV Cache Beyond HBM with Lookahead
 * Sparse Prefetching) keeps only the most relevant KV blocks of each KV head in
 * HBM during decode, predicts them with the queries of lookahead (speculative
 * draft) tokens, and prefetches the missing ones from a host-memory tier under
 * a per-step cap.  One layer-step of the hot path is five calls, in order:
 *
 *   oasis_score_blocks       score every KV block against the lookahead queries
 *   oasis_topk_select        keep the Kb best blocks (the token budget)
 *   oasis_fetch_diff_capped  pick the best selected-but-missing blocks, <= cap
 *   oasis_gather_h2d         copy them host -> HBM slots, update the tables
 *   oasis_sparse_decode_attn attention of the true queries over the resident
 *                            selected blocks
 *
 * Conventions for every call
 *   - Buffers are caller-owned.  "device" pointers are CUDA device memory (or
 *     any pointer the GPU may dereference); "host" pointers are plain CPU memory.
 *     The library allocates nothing and frees nothing.
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL means the
 *     legacy default stream) and returns after enqueueing its kernels.
 *   - Shapes and pointers are validated synchronously: a bad argument returns
 *     OASIS_ERR_INVALID (or OASIS_ERR_UNSUPPORTED for a shape outside the
 *     supported range) and launches nothing.  A failed launch returns
 *     OASIS_ERR_CUDA.  oasis_last_error() describes the last failure of the
 *     calling thread.
 *   - Device-side problems that only the kernels can see (an index out of
 *     range in a table) are OR-ed into a caller-provided uint32 error word
 *     (OASIS_EW_* bits); the offending entry is skipped, nothing faults.
 *   - bf16 tensors hold IEEE bfloat16 bit patterns; all inputs must be finite.
 *   - Layer slicing is done by the caller through pointer offsets; every
 *     per-layer tensor below is described for one layer.
 *
 * Shape (oasis_shape):
 *   B      requests in the batch               (1 .. 65535)
 *   Hq     query heads                          Hq = G * Hkv, G in {1,2,4,8}
 *   Hkv    KV heads
 *   d      head dimension                       must be 128
 *   bs     tokens per KV block                  must be 16
 *   nb_max blocks per (request, KV head) in the key cache, the host tier and
 *          blk2slot                             (1 .. 8192)
 *   n_la   lookahead queries per request        n_la * G <= 32
 *   Kb     token budget in blocks               (1 .. 256)
 *   P      HBM slots per (request, KV head)     Kb <= P <= 1024
 *
 * Context lengths: ctx_len[b] (device int32 [B]) is the number of valid tokens
 * of request b; request b has nb_b = ceil(ctx_len[b] / bs) blocks (clamped to
 * nb_max).  Tokens t >= ctx_len[b] are never scored or attended.
 */
#ifndef OASIS_H_
#define OASIS_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define OASIS_API __attribute__((visibility("default")))
#else
#define OASIS_API
#endif

struct CUstream_st;
/* Same type as cudaStream_t; NULL selects the legacy default stream. */
typedef struct CUstream_st* oasis_stream_t;

typedef enum oasis_status {
  OASIS_OK = 0,
  OASIS_ERR_INVALID = 1,      /* bad pointer, size or shape; nothing launched   */
  OASIS_ERR_CUDA = 2,         /* a CUDA runtime call or launch failed            */
  OASIS_ERR_TIMEOUT = 3,      /* a bounded wait gave up                          */
  OASIS_ERR_UNSUPPORTED = 4   /* valid but outside the supported shape range     */
} oasis_status;

/* Bits OR-ed into the device error word by the kernels. */
#define OASIS_EW_BAD_BLOCK 0x1u  /* a block index outside [0, nb_max)            */
#define OASIS_EW_BAD_SLOT 0x2u   /* a slot index outside [0, P)                  */
#define OASIS_EW_NO_SLOT 0x4u    /* more blocks to fetch than candidate slots    */
#define OASIS_EW_BAD_COUNT 0x8u  /* nsel / nfetch outside its range              */
#define OASIS_EW_TIMEOUT 0x10u   /* a bounded wait on a host flag gave up        */

typedef struct oasis_shape {
  int32_t B, Hq, Hkv, d, bs, nb_max, n_la, Kb, P;
} oasis_shape;

/* Library version string, e.g. "oasis-gb300 0.1 sm_103a". */
OASIS_API const char* oasis_version(void);

/* Description of the last non-OK status returned on the calling thread. */
OASIS_API const char* oasis_last_error(void);

/*
 * a1. Block scoring.
 * Defines: the lookahead prediction of the next step's important KV blocks
 * (OasisKV pages: abstract; metalmedia.ai page, explanatory figure step 2 and
 * Figure 7 caption, where the draft queries are matched against the keys to
 * choose next step's top-K blocks).  The block score is the exact form of that
 * match:
 *   score[b][h][x] = max over j < n_la, g < G, t in block x with t < ctx_len[b]
 *                    of  q_la[b][j][h*G + g] . k[b][h][t] / sqrt(d).
 * Arguments:
 *   k_hbm     device bf16 [B][Hkv][nb_max*bs][d]  keys of one layer (row-major)
 *   ctx_len   device int32 [B]
 *   q_la      device bf16 [B][n_la][Hq][d]        lookahead queries of the layer
 *   scores    device float [B][Hkv][nb_max][2]    out: for every block x < nb_b,
 *             scores[..][x][0] = an approximation s~ of score(x) computed on the
 *             tensor cores, scores[..][x][1] = a bound e with |s~ - score| <= e.
 *             Entries x >= nb_b are not written.
 *   err_word  device uint32 [1] or NULL; OR-ed with OASIS_EW_TIMEOUT if a
 *             bounded wait inside the kernel gave up (the scores are then
 *             incomplete).
 * The bound is e = 2^-12 * max_n |q_n|_2 * max_t |k_t|_2 / sqrt(d) (plus the
 * rounding of the 1/sqrt(d) product); it is an upper bound on the error of
 * fp32-accumulated bf16 products with a wide margin.  Selection never trusts
 * s~ inside this interval: it re-scores those blocks exactly.
 * Two kernels implement it: by default a tcgen05/TMA/TMEM kernel (two CTAs per
 * SM, each a TMA producer, a single-thread MMA issuer and two groups of epilogue
 * warps); after oasis_set_option(OASIS_OPT_SCORE_KERNEL, OASIS_SCORE_KERNEL_MMA)
 * warp-level mma.sync tiles fed by direct 16-byte loads (also used for shapes
 * whose layer has more than 2^31 - 1 key rows).  Their s~ may differ inside the
 * bound; everything selection derives from them is identical.
 */
OASIS_API oasis_status oasis_score_blocks(const oasis_shape* shape, const void* k_hbm,
                                const int32_t* ctx_len, const void* q_la,
                                float* scores, uint32_t* err_word, oasis_stream_t stream);

/*
 * a1, with work handed out at run time: the same scores as oasis_score_blocks
 * (the mma.sync kernel, same bound), but only part of the valid blocks
 * (OASIS_OPT_SCORE_STATIC_SHARE, 75% by default) is split into fixed equal shares
 * as oasis_score_blocks splits all of them; thread blocks then take chunks of 64
 * blocks of the rest from an atomic counter, so thread blocks that start late -
 * because kernels of other streams still hold their SMs - take fewer chunks
 * rather than finishing last.  The grid leaves `reserve_ctas`
 * thread-block slots of the GPU unused, room for such kernels.
 * Arguments: as oasis_score_blocks, plus
 *   work          device uint32 [2], 8-byte aligned: must be zero before the
 *                 call; the last thread block to finish sets it back to zero, so
 *                 it is ready for the next call.  Calls that may overlap on the
 *                 GPU need different work words; a call that does not complete
 *                 (an error) can leave it non-zero.
 *   reserve_ctas  0 .. 4096 thread-block slots (of 128 threads, about 16K
 *                 registers each) left free
 * There is no error word: nothing here can fail once launched.
 */
OASIS_API oasis_status oasis_score_blocks_dynamic(const oasis_shape* shape, const void* k_hbm,
                                                  const int32_t* ctx_len, const void* q_la,
                                                  float* scores, uint32_t* work,
                                                  int32_t reserve_ctas, oasis_stream_t stream);

/*
 * a2. Top-K under the token budget.
 * Defines: keep, per KV head, the Kb highest-scoring blocks (OasisKV pages:
 * abstract, 2,048-token KV budget; Figure 7 caption, top-K blocks).
 *   S = the min(Kb, nb_b) blocks ranked first by (exact score descending,
 *       block index ascending).
 * Blocks whose score interval from oasis_score_blocks straddles the selection
 * boundary are re-scored exactly (integer arithmetic on the bf16 products), so
 * S is exactly the set the definition gives.
 * Arguments:
 *   scores    device float [B][Hkv][nb_max][2]  from oasis_score_blocks
 *   k_hbm, q_la, ctx_len                         the same tensors as for scoring
 *   sel       device int32 [B][Hkv][Kb]          out: S in ascending block order,
 *                                                entries >= nsel are set to -1
 *   nsel      device int32 [B][Hkv]              out: |S| = min(Kb, nb_b)
 */
OASIS_API oasis_status oasis_topk_select(const oasis_shape* shape, const float* scores,
                               const void* k_hbm, const void* q_la,
                               const int32_t* ctx_len, int32_t* sel, int32_t* nsel,
                               oasis_stream_t stream);

/*
 * a3. Capped diff against the HBM-resident set.
 * Defines: compare the predicted set with the blocks already in HBM, fetch only
 * the missing ones, at most a per-step cap (metalmedia.ai page, explanatory
 * figure step 3; Table 2 caption, where a fetch ratio limits how many blocks
 * one step may fetch).
 *   M = { x in S : blk2slot[x] == -1 },
 *   F = the min(fetch_cap, |M|) blocks of M ranked first by (exact score
 *       descending, block index ascending), emitted in ascending block order.
 * Arguments:
 *   scores, k_hbm, q_la, ctx_len   as for oasis_topk_select (exact re-scoring)
 *   sel, nsel                      from oasis_topk_select
 *   blk2slot  device int32 [B][Hkv][nb_max]  slot of each resident block, -1 if
 *                                             not resident (read only)
 *   fetch_cap blocks per (request, KV head), 0 <= fetch_cap <= Kb
 *   fetch     device int32 [B][Hkv][Kb]       out: F, entries >= nfetch are -1
 *   nfetch    device int32 [B][Hkv]           out: |F|
 */
OASIS_API oasis_status oasis_fetch_diff_capped(const oasis_shape* shape, const float* scores,
                                     const void* k_hbm, const void* q_la,
                                     const int32_t* ctx_len, const int32_t* sel,
                                     const int32_t* nsel, const int32_t* blk2slot,
                                     int32_t fetch_cap, int32_t* fetch, int32_t* nfetch,
                                     oasis_stream_t stream);

/*
 * a2 + a3 in one launch: oasis_topk_select followed by oasis_fetch_diff_capped on
 * the selection it wrote, run by the same thread block of each (request, KV head).
 * Arguments are the union of the two calls'; outputs (sel, nsel, fetch, nfetch)
 * are exactly those of the two calls made one after the other.  host_kv, if not
 * NULL (the mapped host tier as for oasis_gather_h2d), makes each fetched block's
 * 8 KiB be prefetched into L2 as soon as F is known, so a gather right after
 * finds it there; it changes no output.
 * oasis_topk_select_diff_pooled: the same with the pooled score (f1 below).
 */
OASIS_API oasis_status oasis_topk_select_diff(const oasis_shape* shape, const float* scores,
                                              const void* k_hbm, const void* q_la,
                                              const int32_t* ctx_len, const int32_t* blk2slot,
                                              int32_t fetch_cap, int32_t* sel, int32_t* nsel,
                                              int32_t* fetch, int32_t* nfetch, const void* host_kv,
                                              oasis_stream_t stream);

OASIS_API oasis_status oasis_topk_select_diff_pooled(const oasis_shape* shape,
                                                     const float* scores, const void* k_pooled,
                                                     const void* q_la, const int32_t* ctx_len,
                                                     const int32_t* blk2slot, int32_t fetch_cap,
                                                     int32_t* sel, int32_t* nsel, int32_t* fetch,
                                                     int32_t* nfetch, const void* host_kv,
                                                     oasis_stream_t stream);

/*
 * a4. Host-tier gather into HBM slots, with the head-wise block table update.
 * Defines: prefetch the selected blocks from the host tier into the limited set
 * of HBM slots (OasisKV abstract; metalmedia.ai page, explanatory figure step 4),
 * the head-wise table from GPU blocks to host-tier blocks (Figure 9 caption) and
 * LRU eviction (Table 2 caption).
 *   Candidate slots, per (request, KV head): the free slots (slot2blk == -1) in
 *   ascending order, then the LRU victims, i.e. the slots whose block is not in
 *   S, ordered by (last_used, block).  F[i] (ascending) takes the i-th
 *   candidate: its K and V are copied from the host tier into that slot, the
 *   evicted block gets blk2slot = -1, and blk2slot/slot2blk are updated.
 *   Finally last_used[slot] = step for every block of S that is resident.
 * Arguments:
 *   host_kv   bf16 [B][Hkv][nb_max][2][bs][d] in page-locked host memory the GPU
 *             can address (cudaHostAlloc / cudaHostRegister, mapped); element
 *             [..][x][0] holds the keys of block x, [..][x][1] its values.  The
 *             kernel reads it with zero-copy loads over the host link.
 *   sel, nsel, fetch, nfetch          from the two calls above
 *   blk2slot  device int32 [B][Hkv][nb_max]   in/out
 *   slot2blk  device int32 [B][Hkv][P]        in/out, -1 = free slot
 *   last_used device int32 [B][Hkv][P]        in/out
 *   step      device int32 [1]: the decode step number written into last_used
 *             (read on the device, so a captured sequence of calls can advance
 *             it without host involvement)
 *   k_pool    device bf16 [B][Hkv][P][bs][d]  in/out (slots written for F)
 *   v_pool    device bf16 [B][Hkv][P][bs][d]  in/out
 *   err_word  device uint32 [1]               OR-ed with OASIS_EW_* bits
 * Requires P >= Kb, so a candidate slot always exists for every block of F.
 */
OASIS_API oasis_status oasis_gather_h2d(const oasis_shape* shape, const void* host_kv,
                              const int32_t* sel, const int32_t* nsel,
                              const int32_t* fetch, const int32_t* nfetch,
                              int32_t* blk2slot, int32_t* slot2blk, int32_t* last_used,
                              const int32_t* step, void* k_pool, void* v_pool,
                              uint32_t* err_word, oasis_stream_t stream);

/*
 * a4, split in two halves so that the host-link copy can leave the critical path
 * (prefetching ahead of use is the point of the method: OasisKV abstract,
 * metalmedia.ai page, Figure 7 caption).  The three calls below together give
 * exactly the tables and pools of oasis_gather_h2d.
 *
 * oasis_assign_slots: the table half of oasis_gather_h2d - candidate slots,
 *   evictions, the new blk2slot/slot2blk entries and the LRU clock - with the
 *   same arguments minus host_kv, k_pool and v_pool.  The pools are not touched:
 *   until the data half has run, the slots assigned to F hold stale data.
 */
OASIS_API oasis_status oasis_assign_slots(const oasis_shape* shape, const int32_t* sel,
                                          const int32_t* nsel, const int32_t* fetch,
                                          const int32_t* nfetch, int32_t* blk2slot,
                                          int32_t* slot2blk, int32_t* last_used,
                                          const int32_t* step, uint32_t* err_word,
                                          oasis_stream_t stream);

/*
 * oasis_copy_fetched: the data half.  For every entry x = fetch[b][h][i],
 *   i < nfetch[b][h], copies K and V of block x from host_kv into slot
 *   blk2slot[b][h][x] of k_pool/v_pool.  It must run after the
 *   oasis_assign_slots call of the same fetch list and before anything reads
 *   those slots.  An entry whose block has no slot (-1) is skipped; a block or
 *   slot index out of range sets OASIS_EW_BAD_BLOCK / OASIS_EW_BAD_SLOT.
 * Arguments:
 *   host_kv        as for oasis_gather_h2d (mapped page-locked host memory)
 *   fetch, nfetch  from oasis_fetch_diff_capped (read only)
 *   blk2slot       device int32 [B][Hkv][nb_max] after oasis_assign_slots (read only)
 *   k_pool, v_pool device bf16 [B][Hkv][P][bs][d]   slots of F written
 *   err_word       device uint32 [1], required
 */
OASIS_API oasis_status oasis_copy_fetched(const oasis_shape* shape, const void* host_kv,
                                          const int32_t* fetch, const int32_t* nfetch,
                                          const int32_t* blk2slot, void* k_pool, void* v_pool,
                                          uint32_t* err_word, oasis_stream_t stream);

/*
 * oasis_copy_fetched_wait: oasis_copy_fetched that first waits, with a bounded
 *   number of polls, for a host-written ready flag.  A host-side producer that
 *   fills the host tier (a slower tier, a remote fetch, the compensating fetch
 *   after a misprediction that the limitations list on the metalmedia.ai page
 *   mentions) writes the data, then sets *ready_flag >= ready_value; the copy
 *   reads the blocks only after it sees that.  Each thread block polls the flag
 *   (relaxed system-scope loads about 256 ns apart) at most max_polls times;
 *   if the flag is still below ready_value it sets OASIS_EW_TIMEOUT in err_word
 *   and copies nothing, so no kernel is left waiting whatever the host does.
 *   The pools' slots of F then keep their old contents (the table half has
 *   already mapped them): the caller must not attend them before a copy
 *   succeeds.  The call itself returns OASIS_OK once enqueued; read the outcome
 *   with oasis_error_word_status.
 * Arguments: as oasis_copy_fetched, plus
 *   ready_flag   uint32 in page-locked, device-mapped host memory (cudaHostAlloc
 *                mapped / cudaHostRegister mapped), 4-byte aligned
 *   ready_value  the copy proceeds once *ready_flag >= ready_value
 *   max_polls    1 .. OASIS_MAX_READY_POLLS (about max_polls x 0.25-0.5 us)
 */
#define OASIS_MAX_READY_POLLS (1 << 22)
OASIS_API oasis_status oasis_copy_fetched_wait(const oasis_shape* shape, const void* host_kv,
                                               const int32_t* fetch, const int32_t* nfetch,
                                               const int32_t* blk2slot, void* k_pool, void* v_pool,
                                               const uint32_t* ready_flag, uint32_t ready_value,
                                               int32_t max_polls, uint32_t* err_word,
                                               oasis_stream_t stream);

/*
 * oasis_error_word_status: waits for `stream` (cudaStreamSynchronize), reads the
 *   device error word and returns OASIS_ERR_TIMEOUT if OASIS_EW_TIMEOUT is set
 *   (a bounded wait gave up), else OASIS_OK; *bits (may be NULL) receives the
 *   whole word.  A blocking call: use it outside the decode loop's hot path or
 *   after a step, not between the launches of one.
 */
OASIS_API oasis_status oasis_error_word_status(const uint32_t* err_word, oasis_stream_t stream,
                                               uint32_t* bits);

/*
 * oasis_score_blocks_copy: oasis_score_blocks of one layer and
 *   oasis_copy_fetched of another (the copy arguments may belong to any layer
 *   of the same shape; they must not alias k_hbm, q_la or scores) in one launch.
 *   Each warp stages its first fetched block from the host before it scores and
 *   writes it to the slot after, so the host-link latency overlaps the HBM-bound
 *   scoring.  Results are those of the two calls made one after the other.
 *   err_word is required (it receives both calls' bits).  With the tcgen05
 *   scorer selected (OASIS_OPT_SCORE_KERNEL) the two are launched one after the
 *   other instead.
 */
OASIS_API oasis_status oasis_score_blocks_copy(const oasis_shape* shape, const void* k_hbm,
                                               const int32_t* ctx_len, const void* q_la,
                                               float* scores, const void* host_kv,
                                               const int32_t* fetch, const int32_t* nfetch,
                                               const int32_t* blk2slot, void* k_pool,
                                               void* v_pool, uint32_t* err_word,
                                               oasis_stream_t stream);

/*
 * a5. Block-sparse paged decode attention.
 * Defines: decode attention of the next-token queries over only the resident
 * selected KV blocks (OasisKV abstract; Figure 7 caption, right).
 *   A = { x in S : blk2slot[x] != -1 }, and for every query head hq = h*G + g
 *   out[b][hq] = sum over valid tokens t of A of softmax_t(scale * q.k_t) v_t,
 *   or zero when A has no valid token.
 * Arguments:
 *   q         device bf16 [B][Hq][d]            true (next-token) queries
 *   k_pool, v_pool  device bf16 [B][Hkv][P][bs][d]
 *   sel, nsel, blk2slot, ctx_len               as above
 *   scale     softmax scale, normally 1/sqrt(d)
 *   workspace device scratch of ws_bytes >= oasis_attn_workspace_bytes(shape);
 *             contents on entry are ignored; not touched by other calls
 *   out       device float [B][Hq][d]           out
 * Split-K: the blocks of each head are cut into chunks attended by separate
 * thread blocks; a second kernel merges the partial softmax states.
 */
OASIS_API oasis_status oasis_sparse_decode_attn(const oasis_shape* shape, const void* q,
                                      const void* k_pool, const void* v_pool,
                                      const int32_t* sel, const int32_t* nsel,
                                      const int32_t* blk2slot, const int32_t* ctx_len,
                                      float scale, void* workspace, size_t ws_bytes,
                                      float* out, oasis_stream_t stream);

/*
 * Token append (long-output decode).
 * Defines: decode grows each request's KV cache by one token per step (OasisKV
 * abstract; metalmedia.ai page, Table 1 "long output" rows and Figure 11
 * caption).  For every request b with t = ctx_len[b] < nb_max*bs, and every KV
 * head h, the new key/value row is written to
 *   k_hbm[b][h][t], host_kv[b][h][t/bs][0][t%bs] (key), host_kv[..][1][t%bs]
 *   (value), and, when blk2slot[b][h][t/bs] = p >= 0, to k_pool/v_pool[b][h][p][t%bs];
 * then, if `advance` is nonzero, ctx_len[b] = t + 1.  A model with several
 * layers calls this once per layer with the same ctx_len and advance = 1 on the
 * last call only.  A full cache (t >= nb_max*bs) sets OASIS_EW_BAD_COUNT and
 * leaves request b unchanged.
 * Arguments:
 *   k_new, v_new  device bf16 [B][Hkv][d]      the new token's key and value
 *   ctx_len       device int32 [B]             in/out
 *   k_hbm         device bf16 [B][Hkv][nb_max*bs][d]   in/out
 *   host_kv       page-locked mapped host memory, layout as in oasis_gather_h2d
 *   blk2slot      device int32 [B][Hkv][nb_max]        read only
 *   k_pool, v_pool device bf16 [B][Hkv][P][bs][d]      in/out
 *   err_word      device uint32 [1] or NULL
 */
OASIS_API oasis_status oasis_append_kv(const oasis_shape* shape, const void* k_new, const void* v_new,
                                       int32_t* ctx_len, void* k_hbm, void* host_kv,
                                       const int32_t* blk2slot, void* k_pool, void* v_pool,
                                       int32_t advance, uint32_t* err_word, oasis_stream_t stream);

/* Bytes of device workspace oasis_sparse_decode_attn needs for `shape` (0 on a bad shape). */
OASIS_API size_t oasis_attn_workspace_bytes(const oasis_shape* shape);

/*
 * Allocation-free attention.  The pages have no counterpart: this is a calling
 * convenience of this library, not a step of the method.
 *
 * Same operation, arguments, output and error behaviour as
 * oasis_sparse_decode_attn, minus the workspace: the split-K scratch lives in a
 * device array built into the library (OASIS_ATTN_NOALLOC_MAX_WORKSPACE_BYTES
 * on every GPU that loads it, held until the process exits).  It is for callers
 * that cannot allocate device memory when they call - a serving loop whose
 * device-memory budget is fixed at start-up, or host code that must not call
 * cudaMalloc on its decode path because that call can block on the device.
 *   - It allocates nothing: no cudaMalloc/cudaFree or allocating library call.
 *   - The first call on a device looks up the array's device address once for
 *     that device (cudaGetSymbolAddress, with the device current); make that
 *     first call before any stream capture.
 *   - Shapes whose scratch (oasis_attn_workspace_bytes) exceeds the array are
 *     rejected with OASIS_ERR_UNSUPPORTED and a message in oasis_last_error().
 *   - Every call on a device shares the one array, whose contents persist
 *     between calls; two calls whose kernels overlap on the GPU (different
 *     streams without ordering) race on it and produce wrong outputs.  Order
 *     such calls, or use oasis_sparse_decode_attn with separate workspaces.
 *   - The array's address is cached per device for the life of the process.
 *     cudaDeviceReset destroys the context that holds it, so the cached address
 *     is stale afterwards: do not use this call in a process after a
 *     cudaDeviceReset of that device (use oasis_sparse_decode_attn instead).
 */
#define OASIS_ATTN_NOALLOC_MAX_WORKSPACE_BYTES (8u << 20)
OASIS_API oasis_status oasis_sparse_decode_attn_noalloc(const oasis_shape* shape, const void* q,
                                                        const void* k_pool, const void* v_pool,
                                                        const int32_t* sel, const int32_t* nsel,
                                                        const int32_t* blk2slot, const int32_t* ctx_len,
                                                        float scale, float* out, oasis_stream_t stream);

/*
 * f1. Scoring from min/max pooled compressed keys.
 * Defines: the GPU keeps, besides the sparse working set, compressed keys made by
 * per-block min/max pooling, and the draft query scans those to predict the next
 * step's top-K blocks (metalmedia.ai page, Figure 7 caption, left).  The pooled
 * score of block x is the largest value a key inside the block's per-dimension
 * [lo, hi] box can give:
 *   pooled(x) = max over j < n_la, g < G of
 *               sum_i max(q_la[b][j][h*G+g][i] * hi[x][i], q_la[..][i] * lo[x][i]) / sqrt(d),
 *   hi[x][i] / lo[x][i] = max / min over the valid tokens t of x of k[t][i].
 * It bounds the max-dot score of a1 from above and equals it for a block with one
 * valid token.  Ranking, ties, S and F are as for a2/a3 with this score.
 *
 * k_pooled: device bf16 [B][Hkv][nb_max][2][d]: row 0 = hi, row 1 = lo; blocks
 * without a valid token hold zeros.  512 bytes per block.
 *
 * oasis_pool_keys: builds k_pooled for every block from k_hbm (layout as for
 *   oasis_score_blocks) and ctx_len.
 * oasis_pool_append: folds k_new (device bf16 [B][Hkv][d]) into the block of
 *   token position ctx_len[b] (a block's first token sets both rows).  Call it
 *   with the same ctx_len as the oasis_append_kv of that token, before that
 *   call advances ctx_len.  A position outside [0, nb_max*bs) sets
 *   OASIS_EW_BAD_COUNT in err_word (may be NULL) and is skipped.
 * oasis_score_blocks_pooled: writes scores exactly as oasis_score_blocks does
 *   (approximation and certified bound; here e = 2^-12 |q| |k'| / sqrt(d) + ...,
 *   |k'|^2 = |hi|^2 + |lo|^2), reading 512 bytes per block.  If host_kv is not
 *   NULL the launch also carries oasis_copy_fetched(host_kv, fetch, nfetch,
 *   blk2slot, k_pool, v_pool, err_word) as oasis_score_blocks_copy does (err_word
 *   then required); with host_kv NULL those five pointers are ignored.
 * oasis_topk_select_pooled / oasis_fetch_diff_capped_pooled: as a2 / a3 with the
 *   pooled score; k_pooled takes the place of k_hbm for the exact re-scoring.
 */
OASIS_API oasis_status oasis_pool_keys(const oasis_shape* shape, const void* k_hbm,
                                       const int32_t* ctx_len, void* k_pooled,
                                       oasis_stream_t stream);

OASIS_API oasis_status oasis_pool_append(const oasis_shape* shape, const void* k_new,
                                         const int32_t* ctx_len, void* k_pooled,
                                         uint32_t* err_word, oasis_stream_t stream);

OASIS_API oasis_status oasis_score_blocks_pooled(const oasis_shape* shape, const void* k_pooled,
                                                 const int32_t* ctx_len, const void* q_la,
                                                 float* scores, const void* host_kv,
                                                 const int32_t* fetch, const int32_t* nfetch,
                                                 const int32_t* blk2slot, void* k_pool,
                                                 void* v_pool, uint32_t* err_word,
                                                 oasis_stream_t stream);

OASIS_API oasis_status oasis_topk_select_pooled(const oasis_shape* shape, const float* scores,
                                                const void* k_pooled, const void* q_la,
                                                const int32_t* ctx_len, int32_t* sel,
                                                int32_t* nsel, oasis_stream_t stream);

OASIS_API oasis_status oasis_fetch_diff_capped_pooled(const oasis_shape* shape,
                                                      const float* scores, const void* k_pooled,
                                                      const void* q_la, const int32_t* ctx_len,
                                                      const int32_t* sel, const int32_t* nsel,
                                                      const int32_t* blk2slot,
                                                      int32_t fetch_cap, int32_t* fetch,
                                                      int32_t* nfetch, oasis_stream_t stream);

/*
 * f2. Fused look-ahead attention.
 * Defines: the attention kernel processes the normal and the draft queries
 * together over the sparse KV (metalmedia.ai page, Figure 7 caption, right).
 * With A as in oasis_sparse_decode_attn, for every query head hq = h*G + g:
 *   out[b][hq]       = sum over valid tokens t of A of softmax_t(scale * q[b][hq] . k_t) v_t
 *   out_la[b][j][hq] = the same with q_la[b][j][hq] (j < n_la),
 * zero where A has no valid token.  Each attended block's K and V are read once
 * per 16 query rows ((1 + n_la) * G rows per KV head).
 * Arguments: as oasis_sparse_decode_attn, plus
 *   q_la      device bf16 [B][n_la][Hq][d]   the lookahead queries
 *   out_la    device float [B][n_la][Hq][d]  out
 *   workspace ws_bytes >= oasis_attn_lookahead_workspace_bytes(shape)
 */
OASIS_API size_t oasis_attn_lookahead_workspace_bytes(const oasis_shape* shape);

OASIS_API oasis_status oasis_sparse_decode_attn_lookahead(const oasis_shape* shape, const void* q,
                                                          const void* q_la, const void* k_pool,
                                                          const void* v_pool, const int32_t* sel,
                                                          const int32_t* nsel,
                                                          const int32_t* blk2slot,
                                                          const int32_t* ctx_len, float scale,
                                                          void* workspace, size_t ws_bytes,
                                                          float* out, float* out_la,
                                                          oasis_stream_t stream);

/*
 * Host-tier warm-up (the pages have no counterpart: a platform utility).
 * oasis_touch_host: reads every byte of [host_ptr, host_ptr + bytes) once with
 * the SMs' zero-copy loads and discards the data.  On the GB300 systems this
 * library was measured on, the first SM reads into some regions of a large
 * page-locked allocation stall for milliseconds until the region has been read
 * once (copy-engine transfers do not clear this); calling this after filling the
 * host tier keeps those stalls out of the gathers.  host_ptr: page-locked,
 * device-mapped host memory (as host_kv), 16-byte aligned; bytes a multiple of
 * 16; sink: device uint32 or NULL (written only in a case that does not occur).
 * Asynchronous on stream; a 100 GiB tier takes about half a second.
 */
OASIS_API oasis_status oasis_touch_host(const void* host_ptr, size_t bytes, uint32_t* sink,
                                        oasis_stream_t stream);

/*
 * Process-wide launch options (the pages have no counterpart: scheduling knobs).
 * OASIS_OPT_SCORE_CTAS_PER_SM: the mma.sync max-dot block scorer (with or without
 *   a carried copy) sizes its persistent grid to value CTAs per SM (0 = as many as
 *   fit, the default); so does the pooled scorer (4 CTAs of 4 warps per SM when
 *   0).  A caller that runs the selection, gather and attention kernels of one
 *   layer beside the scorer of the next on another stream leaves them room this
 *   way.  Read at every launch; results do not depend on it.
 * Unknown options or values return OASIS_ERR_INVALID.
 */
#define OASIS_OPT_SCORE_CTAS_PER_SM 1
/*
 * OASIS_OPT_SCORE_KERNEL: which kernel oasis_score_blocks (and
 *   oasis_score_blocks_copy) launches: OASIS_SCORE_KERNEL_TC (TMA + tcgen05 +
 *   TMEM, the default) or OASIS_SCORE_KERNEL_MMA (mma.sync).  Same definition and
 *   bound; selection results do not depend on it.  Read at every scoring call
 *   (an atomic load, no environment lookup).
 */
#define OASIS_OPT_SCORE_KERNEL 2
/*
 * OASIS_OPT_COPY_CTAS: the thread blocks (4 warps each) of oasis_copy_fetched and
 *   oasis_copy_fetched_wait; 0 (the default) = one warp per fetch entry up to four
 *   blocks per SM.  A small value confines the zero-copy host reads to a few SMs
 *   (each warp then streams several entries); results do not depend on it.
 */
#define OASIS_OPT_COPY_CTAS 3
/*
 * OASIS_OPT_SCORE_STATIC_SHARE: the part of oasis_score_blocks_dynamic's work, in
 *   per mille of the valid blocks, split into fixed equal shares before the rest
 *   is handed out in chunks (0 = all in chunks, 1000 = none; default 750).
 *   Read at every launch; results do not depend on it.
 */
#define OASIS_OPT_SCORE_STATIC_SHARE 4
#define OASIS_SCORE_KERNEL_MMA 0
#define OASIS_SCORE_KERNEL_TC 1
OASIS_API oasis_status oasis_set_option(int32_t option, int32_t value);

/*
 * f3. Agreement of a predicted top-K set with the exact one (measurement only).
 * Defines: the per-layer agreement between the blocks the draft (lookahead)
 * queries select and the exact top-K blocks of the true next-token query
 * (metalmedia.ai page, Figure 6 caption; at K = 20 with the previous token as
 * the predictor, Figure 4 caption).  Obtain the exact set with
 * oasis_score_blocks + oasis_topk_select on a shape with n_la = 1 and the true
 * queries [B][Hq][d] as q_la; the predicted set is oasis_topk_select's output.
 *   counts[b][h][0] = |pred & exact|
 *   counts[b][h][1] = |pred & exact & resident| (resident: blk2slot >= 0), or -1
 *                     when blk2slot is NULL
 *   counts[b][h][2] = |exact|
 * Arguments:
 *   pred, npred    device int32 [B][Hkv][Kb], [B][Hkv]  ascending block lists
 *   exact, nexact  device int32 [B][Hkv][Kb], [B][Hkv]  ascending block lists
 *   blk2slot       device int32 [B][Hkv][nb_max] or NULL
 *   counts         device int32 [B][Hkv][3]             out
 *   err_word       device uint32 [1] or NULL (OASIS_EW_BAD_COUNT / _BAD_BLOCK)
 * Only shape.B, Hkv, Kb and nb_max are used; the other fields are checked as
 * for every call.  Unsorted pred gives wrong counts but never reads out of
 * bounds.
 */
OASIS_API oasis_status oasis_set_agreement(const oasis_shape* shape, const int32_t* pred,
                                           const int32_t* npred, const int32_t* exact,
                                           const int32_t* nexact, const int32_t* blk2slot,
                                           int32_t* counts, uint32_t* err_word,
                                           oasis_stream_t stream);

/*
 * Kernel span trace (diagnostics; the pages have no counterpart).  With a trace
 * buffer set, thread 0 of every thread block of the kernels below reads the GPU's
 * nanosecond global timer when the block starts and when it ends, and each launch
 * gets one record: the earliest start and the latest end over its blocks.  A
 * CUDA graph replays without event nodes between its kernels, so the records
 * show where a replayed decode step spends its time without perturbing it.
 *
 * Kinds (record arrays):
 *   OASIS_TRACE_SCORE        max-dot scorers (mma.sync, dynamic, copy-carrying, tcgen05)
 *   OASIS_TRACE_SCORE_POOLED pooled-key scorer
 *   OASIS_TRACE_SELECT       top-K (+ diff) and diff-only selection kernels
 *   OASIS_TRACE_GATHER       gather_h2d (slot assignment, with or without the copy)
 *   OASIS_TRACE_COPY         copy of fetched blocks (oasis_copy_fetched[_wait])
 *   OASIS_TRACE_ATTN         attention partial kernel (its combine launch is not traced)
 *   OASIS_TRACE_APPEND       token append
 * Buffer (caller-owned device memory of oasis_trace_bytes(capacity) bytes, zeroed
 * by the caller before it is set):
 *   uint32 ctl[2 * OASIS_TRACE_KINDS]   per kind: records begun, blocks finished
 *   (padding to 128 bytes)
 *   uint64 rec[OASIS_TRACE_KINDS][capacity][2]
 *     rec[k][i][0] = ~(earliest start in ns), rec[k][i][1] = latest end in ns of
 *     the i-th launch of kind k (modulo capacity); unused records are zero.
 * oasis_trace_set(buf, capacity) makes later launches record into buf; NULL turns
 * tracing off.  The pointer is read when a kernel is launched, so a CUDA graph
 * captured while it is set keeps recording into that buffer on every replay.
 * Records are not cleared when the index wraps: give the buffer the capacity of
 * the launches made between two zeroings.  Launches of one kind that overlap in
 * time share one record.  The buffer must
 * stay allocated while any launch or graph that records into it may run.
 * Errors: capacity < 1 or a buffer not 16-byte aligned -> OASIS_ERR_INVALID.
 */
#define OASIS_TRACE_KINDS 7
#define OASIS_TRACE_SCORE 0
#define OASIS_TRACE_SCORE_POOLED 1
#define OASIS_TRACE_SELECT 2
#define OASIS_TRACE_GATHER 3
#define OASIS_TRACE_COPY 4
#define OASIS_TRACE_ATTN 5
#define OASIS_TRACE_APPEND 6
OASIS_API size_t oasis_trace_bytes(int32_t capacity);
OASIS_API oasis_status oasis_trace_set(void* dev_buf, int32_t capacity);

#ifdef __cplusplus
}
#endif

#endif /* OASIS_H_ */
