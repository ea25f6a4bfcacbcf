// a4: slot assignment, zero-copy host-tier gather into HBM slots, table update.
//
// OasisKV abstract (prefetch from a higher-capacity tier into HBM before the next
// decode step uses the blocks); metalmedia.ai page, Figure 9 caption (a head-wise
// table maps each GPU block of the bounded working set to a CPU block) and
// Table 2 caption (LRU eviction).
//
// One thread block per (request, KV head):
//   1. candidate slots = free slots ascending, then victims (resident blocks not
//      in S) by (last_used, block) - each slot computes its own rank by counting;
//   2. F[i] takes candidate i: evicted block -> blk2slot = -1, then the new
//      mapping is written (evicted blocks are outside S, fetched ones inside, so
//      the two sets of writes never touch the same entry);
//   3. last_used = step for every resident block of S;
//   4. the 8 KiB (K 4 KiB + V 4 KiB) of every fetched block is read from mapped
//      page-locked host memory with 16-byte loads (several in flight per thread)
//      and written to its slot.  The first round of host reads is issued right
//      after the fetch list arrives, before the slot bookkeeping, so the link's
//      latency overlaps it; all table reads happen in one round of loads and the
//      LRU clock is set from shared memory.  The copy is bound by the host link.
// Out-of-range indices set bits of the error word and are skipped.
//
// The same kernel without step 4 is the table half alone (oasis_assign_slots);
// the data half then runs later as a warp-level copy (fetch_copy.cuh), either
// carried by the next layer's block scorer or as its own small kernel here.
#include "fetch_copy.cuh"

namespace oasis {

// 128 threads (4 warps, under 48 registers each): the decode step runs this kernel
// on a side stream beside the previous layer's attention, whose 2 CTAs per SM
// (4 warps x 208 registers each) must still fit next to two of these CTAs, or
// attention spills into a second wave.  The copy is bound by the host link, not
// by the threads that issue it.
constexpr int kGatherThreads = 128;
constexpr int kGatherUnroll = 4;

__device__ __forceinline__ uint4 ld_host16(const void* p) {
  uint4 r;
  asm volatile("ld.global.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

template <bool kCopy>
__global__ void __launch_bounds__(kGatherThreads)
gather_h2d_kernel(Shape s, const uint16_t* __restrict__ host_kv, const int* __restrict__ sel,
                  const int* __restrict__ nsel, const int* __restrict__ fetch,
                  const int* __restrict__ nfetch, int* __restrict__ blk2slot,
                  int* __restrict__ slot2blk, int* __restrict__ last_used, const int* __restrict__ step_ptr,
                  uint16_t* __restrict__ k_pool, uint16_t* __restrict__ v_pool,
                  unsigned* __restrict__ err, TraceBuf trace) {
  TraceScope trace_(trace, OASIS_TRACE_GATHER);
  extern __shared__ __align__(16) int gsm[];
  const int Kb = s.Kb, P = s.P;
  int* S = gsm;              // [Kb]
  int* F = S + Kb;           // [Kb]
  int* s2b = F + Kb;         // [P]
  int* lu = s2b + P;         // [P]
  int* cand = lu + P;        // [P]  slot of the i-th candidate, later class per slot
  int* ins = cand + P;       // [P]  1 if the slot's block is in S
  int* scal = ins + P;       // [4]
  const int head = blockIdx.x;
  const long long tb = (long long)head * s.nb_max;
  const long long ts = (long long)head * P;
  constexpr int kUnits = 2 * kBS * kD * 2 / 16;  // 16-byte pieces per block (K then V): 512
  unsigned ew = 0;

  // one round of independent loads: counts, lists, slot tables
  int ns = nsel[head], nf = nfetch[head];
  const int step = *step_ptr;
  for (int i = threadIdx.x; i < Kb; i += blockDim.x) {
    S[i] = sel[(long long)head * Kb + i];
    F[i] = fetch[(long long)head * Kb + i];
  }
  for (int p = threadIdx.x; p < P; p += blockDim.x) {
    s2b[p] = slot2blk[ts + p];
    lu[p] = last_used[ts + p];
  }
  if (ns < 0 || ns > Kb) { ew |= OASIS_EW_BAD_COUNT; ns = ns < 0 ? 0 : Kb; }
  if (nf < 0 || nf > Kb) { ew |= OASIS_EW_BAD_COUNT; nf = nf < 0 ? 0 : Kb; }
  if (threadIdx.x == 0) { scal[0] = 0; scal[1] = 0; }
  __syncthreads();
  // An out-of-range entry of S is flagged but left in place: S is only searched
  // (binary search for resident blocks, which lie in [0, nb_max)), and keeping
  // the value keeps the list ascending, so it can never match or misplace a
  // valid block.  A bad entry of F is cleared: F drives the copies.
  for (int i = threadIdx.x; i < Kb; i += blockDim.x) {
    if (i < ns && (S[i] < 0 || S[i] >= s.nb_max)) ew |= OASIS_EW_BAD_BLOCK;
    if (i < nf && (F[i] < 0 || F[i] >= s.nb_max)) { ew |= OASIS_EW_BAD_BLOCK; F[i] = -1; }
  }
  for (int p = threadIdx.x; p < P; p += blockDim.x)
    if (s2b[p] >= s.nb_max || s2b[p] < -1) { ew |= OASIS_EW_BAD_BLOCK; s2b[p] = -1; }
  __syncthreads();

  // start the first round of host reads now, so the link latency overlaps the table work
  const int total = nf * kUnits;
  uint4 pre[kGatherUnroll];
  if constexpr (kCopy) {
#pragma unroll
    for (int u = 0; u < kGatherUnroll; ++u) {
      const int id = threadIdx.x + u * blockDim.x;
      if (id < total) {
        const int i = id / kUnits, w = id - i * kUnits;
        const int x = F[i];
        if (x >= 0) pre[u] = ld_host16(host_kv + ((tb + x) * 2 * kBS * kD) + (long long)w * 8);
      }
    }
  }

  // 1. classes and candidate ranks: free slots ascending, then victims by (last_used, block)
  for (int p = threadIdx.x; p < P; p += blockDim.x) {
    const int o = s2b[p];
    bool in_s = false;
    if (o >= 0) {  // binary search in S (ascending)
      int lo = 0, hi = ns - 1;
      while (lo <= hi) {
        const int mid = (lo + hi) >> 1;
        const int v = S[mid];
        if (v == o) { in_s = true; break; }
        if (v < o) lo = mid + 1; else hi = mid - 1;
      }
    }
    ins[p] = in_s ? 1 : 0;
    cand[p] = -1;
    if (o < 0) atomicAdd(&scal[0], 1);
    else if (!in_s) atomicAdd(&scal[1], 1);
  }
  __syncthreads();
  const int nfree = scal[0], nvict = scal[1];
  int myrank[(1024 + kGatherThreads - 1) / kGatherThreads];
  int k = 0;
  for (int p = threadIdx.x; p < P; p += blockDim.x, ++k) {
    const int o = s2b[p];
    int r = -1;
    if (o < 0) {
      r = 0;
      for (int q = 0; q < p; ++q) r += (s2b[q] < 0);
    } else if (!ins[p]) {
      r = nfree;
      const int lp = lu[p];
      for (int q = 0; q < P; ++q) {
        const int oq = s2b[q];
        if (oq < 0 || ins[q] || q == p) continue;
        const int lq = lu[q];
        r += (lq < lp) || (lq == lp && oq < o);
      }
    }
    myrank[k] = r;
  }
  __syncthreads();
  k = 0;
  for (int p = threadIdx.x; p < P; p += blockDim.x, ++k)
    if (myrank[k] >= 0 && myrank[k] < P) cand[myrank[k]] = p;
  __syncthreads();

  // 2. assignment: evict, map, LRU clock (all from shared memory)
  const int ncand = nfree + nvict;
  const int ncopy = nf < ncand ? nf : ncand;
  if (nf > ncand) ew |= OASIS_EW_NO_SLOT;
  for (int i = threadIdx.x; i < ncopy; i += blockDim.x) {
    const int p = cand[i];
    if (p < 0) { ew |= OASIS_EW_BAD_SLOT; continue; }  // duplicate entries in slot2blk
    const int old = s2b[p];
    if (old >= 0) blk2slot[tb + old] = -1;
  }
  __syncthreads();
  for (int i = threadIdx.x; i < ncopy; i += blockDim.x) {
    const int p = cand[i];
    const int x = F[i];
    if (p < 0) continue;
    if (x >= 0) {
      blk2slot[tb + x] = p;
      s2b[p] = x;
      lu[p] = step;
    } else {
      s2b[p] = -1;
    }
  }
  for (int p = threadIdx.x; p < P; p += blockDim.x)
    if (ins[p]) lu[p] = step;
  __syncthreads();
  for (int p = threadIdx.x; p < P; p += blockDim.x) {
    slot2blk[ts + p] = s2b[p];
    last_used[ts + p] = lu[p];
  }

  if constexpr (!kCopy) {
    if (ew) atomicOr(err, ew);
    return;
  }
  // 3. copies: first the prefetched round, then the rest in rounds of kGatherUnroll
#pragma unroll
  for (int u = 0; u < kGatherUnroll; ++u) {
    const int id = threadIdx.x + u * blockDim.x;
    if (id < total) {
      const int i = id / kUnits, w = id - i * kUnits;
      if (i < ncopy && F[i] >= 0 && cand[i] >= 0) {
        uint16_t* to = ((w >> 8) ? v_pool : k_pool) + ((ts + cand[i]) * kBS * kD) + (long long)(w & 255) * 8;
        *reinterpret_cast<uint4*>(to) = pre[u];
      }
    }
  }
  for (int base = threadIdx.x + kGatherUnroll * blockDim.x; base < total; base += blockDim.x * kGatherUnroll) {
    uint4 v[kGatherUnroll];
#pragma unroll
    for (int u = 0; u < kGatherUnroll; ++u) {
      const int id = base + u * blockDim.x;
      if (id < total) {
        const int i = id / kUnits, w = id - i * kUnits;
        const int x = F[i];
        if (x >= 0) v[u] = ld_host16(host_kv + ((tb + x) * 2 * kBS * kD) + (long long)w * 8);
      }
    }
#pragma unroll
    for (int u = 0; u < kGatherUnroll; ++u) {
      const int id = base + u * blockDim.x;
      if (id < total) {
        const int i = id / kUnits, w = id - i * kUnits;
        if (i < ncopy && F[i] >= 0 && cand[i] >= 0) {
          uint16_t* to = ((w >> 8) ? v_pool : k_pool) + ((ts + cand[i]) * kBS * kD) + (long long)(w & 255) * 8;
          *reinterpret_cast<uint4*>(to) = v[u];
        }
      }
    }
  }
  if (ew) atomicOr(err, ew);
}

size_t gather_smem_bytes(const Shape& s) { return sizeof(int) * (2 * (size_t)s.Kb + 4 * (size_t)s.P + 4); }

template <bool kCopy>
static cudaError_t launch_gather(const Shape& s, const uint16_t* host_kv, const int* sel, const int* nsel,
                                 const int* fetch, const int* nfetch, int* blk2slot, int* slot2blk,
                                 int* last_used, const int* step, uint16_t* k_pool, uint16_t* v_pool,
                                 unsigned* err, cudaStream_t stream) {
  const size_t smem = gather_smem_bytes(s);
  if (smem > 48 * 1024) {
    static int attr_cache[kMaxDevicesCached] = {};
    cudaError_t e = ensure_dyn_smem((const void*)gather_h2d_kernel<kCopy>, smem, attr_cache);
    if (e != cudaSuccess) return e;
  }
  gather_h2d_kernel<kCopy><<<s.B * s.Hkv, kGatherThreads, smem, stream>>>(
      s, host_kv, sel, nsel, fetch, nfetch, blk2slot, slot2blk, last_used, step, k_pool, v_pool, err, trace_buf());
  return cudaGetLastError();
}

cudaError_t launch_gather_h2d(const Shape& s, const uint16_t* host_kv, const int* sel, const int* nsel,
                              const int* fetch, const int* nfetch, int* blk2slot, int* slot2blk,
                              int* last_used, const int* step, uint16_t* k_pool, uint16_t* v_pool,
                              unsigned* err, cudaStream_t stream) {
  return launch_gather<true>(s, host_kv, sel, nsel, fetch, nfetch, blk2slot, slot2blk, last_used, step, k_pool,
                             v_pool, err, stream);
}

cudaError_t launch_assign_slots(const Shape& s, const int* sel, const int* nsel, const int* fetch,
                                const int* nfetch, int* blk2slot, int* slot2blk, int* last_used, const int* step,
                                unsigned* err, cudaStream_t stream) {
  return launch_gather<false>(s, nullptr, sel, nsel, fetch, nfetch, blk2slot, slot2blk, last_used, step, nullptr,
                              nullptr, err, stream);
}

// The data half on its own: warps of 4-warp CTAs, 8 KiB of staging per warp.
constexpr int kCopyWarps = 4;

// A host-written ready flag that a copy may wait for (the host tier of a layer
// being filled by a host-side producer).  `flag` is the device address of a
// word of page-locked mapped host memory; the wait ends when *flag >= `value`
// or after `max_polls` polls.
struct ReadyWait {
  const unsigned* flag;
  unsigned value;
  int max_polls;
};

// Relaxed system-scope load: sees the host's write to mapped memory.
__device__ __forceinline__ unsigned ld_relaxed_sys(const unsigned* p) {
  unsigned v;
  asm volatile("ld.relaxed.sys.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Thread 0 of the CTA polls the flag (bounded by max_polls, 256 ns apart); the
// CTA learns the outcome through shared memory.  False: the wait gave up, the
// error word has OASIS_EW_TIMEOUT, and the CTA must not copy.
__device__ __forceinline__ bool wait_ready(const ReadyWait& w, unsigned* err) {
  __shared__ int ok;
  if (threadIdx.x == 0) {
    int polls = 0;
    bool ready = ld_relaxed_sys(w.flag) >= w.value;
    while (!ready && ++polls < w.max_polls) {
      __nanosleep(256);
      ready = ld_relaxed_sys(w.flag) >= w.value;
    }
    if (ready) {
      __threadfence_system();  // the host data written before the flag is read after it
    } else if (err) {
      atomicOr(err, OASIS_EW_TIMEOUT);
    }
    ok = ready ? 1 : 0;
  }
  __syncthreads();
  return ok != 0;
}

template <bool kWait>
__global__ void __launch_bounds__(kCopyWarps * 32) copy_fetched_kernel(Shape s, CopyJob job, ReadyWait rw,
                                                                       TraceBuf tb) {
  TraceScope trace_(tb, OASIS_TRACE_COPY);
  extern __shared__ uint4 copy_buf[];
  if constexpr (kWait) {
    if (!wait_ready(rw, job.err)) return;
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint4* buf = copy_buf + warp * (kCopyUnitBytes / 16);
  const long long gwarp = (long long)blockIdx.x * kCopyWarps + warp;
  const long long nwarps = (long long)gridDim.x * kCopyWarps;
  copy_begin(job, s, gwarp, nwarps, buf, lane);
  copy_finish(job, s, gwarp, nwarps, buf, lane);
}

static int copy_grid(const Shape& s) {
  const int fixed = copy_ctas_option();  // a caller may confine the copy to a few SMs
  if (fixed > 0) return fixed;
  // one warp per live entry up to four CTAs per SM; a warp streams any further entries
  const long long items = (long long)s.B * s.Hkv * s.Kb;
  long long ctas = (items + kCopyWarps - 1) / kCopyWarps;
  const long long cap = 4LL * sm_count();
  if (ctas > cap) ctas = cap;
  if (ctas < 1) ctas = 1;
  return (int)ctas;
}

cudaError_t launch_copy_fetched(const Shape& s, const CopyJob& job, cudaStream_t stream) {
  copy_fetched_kernel<false><<<copy_grid(s), kCopyWarps * 32, kCopyWarps * kCopyUnitBytes, stream>>>(
      s, job, ReadyWait{nullptr, 0u, 0}, trace_buf());
  return cudaGetLastError();
}

cudaError_t launch_copy_fetched_wait(const Shape& s, const CopyJob& job, const unsigned* flag, unsigned value,
                                     int max_polls, cudaStream_t stream) {
  copy_fetched_kernel<true><<<copy_grid(s), kCopyWarps * 32, kCopyWarps * kCopyUnitBytes, stream>>>(
      s, job, ReadyWait{flag, value, max_polls}, trace_buf());
  return cudaGetLastError();
}

}  // namespace oasis
