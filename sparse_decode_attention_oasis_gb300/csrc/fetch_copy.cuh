// The data half of the gather: host tier -> HBM slot copy of the fetched blocks,
// done by whole warps through shared memory with cp.async so that it can ride
// inside another kernel.  The block scorer of the next layer carries it: the copy
// is issued when that kernel starts and written out when its scoring is done, so
// the host link's latency hides behind a few hundred microseconds of HBM-bound
// scoring instead of sitting on the critical path (OasisKV abstract: blocks are
// prefetched into HBM before the decode step that uses them).
//
// The slot of every fetched block must already be in blk2slot (the table half of
// the gather, oasis_assign_slots, writes it).  Work items: item k in
// [0, heads * Kb) is fetch entry i = k / heads of head k % heads and is live iff
// i < nfetch[head].  Global warp w of W takes items w, w + W, w + 2W, ...; the
// i-major order spreads the few live entries of a small cap over many warps.
#pragma once

#include "common.cuh"

namespace oasis {

struct CopyJob {
  const uint16_t* host_kv;  // device address of the layer's mapped host tier [heads][nb_max][2][16][128]
  const int* fetch;         // [heads][Kb]
  const int* nfetch;        // [heads]
  const int* blk2slot;      // [heads][nb_max]
  uint16_t* k_pool;         // [heads][P][16][128]
  uint16_t* v_pool;
  unsigned* err;            // error word (may be null)
};

constexpr int kCopyUnitBytes = 2 * kBS * kD * 2;                  // K then V of one block: 8 KiB
constexpr int kCopyChunksPerLane = kCopyUnitBytes / 16 / 32;      // 16
constexpr int kCopyHalfChunks = kBS * kD * 2 / 16;                // 256 chunks of K, then 256 of V

__device__ __forceinline__ void copy_cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void copy_cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void copy_cp_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

// Next live item at or after `k` (steps of `stride`) for the whole warp.  On
// success returns true with head, the fetched block x and k advanced past it.
// Entries naming a block outside [0, nb_max) set OASIS_EW_BAD_BLOCK and are skipped.
__device__ __forceinline__ bool copy_next_item(const CopyJob& j, const Shape& s, long long& k, long long stride,
                                               int lane, int& head, int& x) {
  const int heads = s.B * s.Hkv;
  const long long nitems = (long long)heads * s.Kb;
  while (k < nitems) {
    const long long kk = k + lane * stride;
    int hd = 0, xx = -1;
    bool live = false;
    if (kk < nitems) {
      const int i = (int)(kk / heads);
      hd = (int)(kk - (long long)i * heads);
      const int nf = j.nfetch[hd];
      if (i < nf && i < s.Kb) {
        xx = j.fetch[(long long)hd * s.Kb + i];
        live = true;
        if (xx < 0 || xx >= s.nb_max) {
          if (j.err) atomicOr(j.err, OASIS_EW_BAD_BLOCK);
          live = false;
        }
      }
    }
    const unsigned m = __ballot_sync(0xffffffffu, live);
    if (m) {
      const int src = __ffs(m) - 1;
      head = __shfl_sync(0xffffffffu, hd, src);
      x = __shfl_sync(0xffffffffu, xx, src);
      k += (long long)(src + 1) * stride;
      return true;
    }
    k += 32 * stride;
  }
  return false;
}

// Issue the 8 KiB of block x of `head` into the warp's staging buffer (one group).
__device__ __forceinline__ void copy_stage(const CopyJob& j, const Shape& s, int head, int x, uint32_t buf,
                                           int lane) {
  const uint16_t* src = j.host_kv + ((long long)head * s.nb_max + x) * (kCopyUnitBytes / 2);
#pragma unroll
  for (int m = 0; m < kCopyChunksPerLane; ++m) {
    const int c = lane + 32 * m;
    copy_cp_async16(buf + c * 16, src + c * 8);
  }
  copy_cp_commit();
}

// Wait for the warp's staged block and store it to its slot.  Each lane stores
// exactly the chunks it staged, so no barrier is needed between wait and store.
__device__ __forceinline__ void copy_store(const CopyJob& j, const Shape& s, int head, int x, const uint4* buf,
                                           int lane) {
  copy_cp_wait_all();
  const int slot = j.blk2slot[(long long)head * s.nb_max + x];
  if (slot < 0) return;  // no slot was free (the table half reported it)
  if (slot >= s.P) {
    if (lane == 0 && j.err) atomicOr(j.err, OASIS_EW_BAD_SLOT);
    return;
  }
  const long long base = ((long long)head * s.P + slot) * (kBS * kD);
#pragma unroll
  for (int m = 0; m < kCopyChunksPerLane; ++m) {
    const int c = lane + 32 * m;
    uint16_t* dst = (c < kCopyHalfChunks ? j.k_pool : j.v_pool) + base + (long long)(c & (kCopyHalfChunks - 1)) * 8;
    *reinterpret_cast<uint4*>(dst) = buf[c];
  }
}

// Warp-level copy loop.  copy_begin stages the warp's first live item (if any);
// copy_finish (after the host kernel's own work) stores it and then streams the
// warp's remaining items one at a time.  Both scan from the same start, so no
// state has to be kept between them.
__device__ __forceinline__ void copy_begin(const CopyJob& j, const Shape& s, long long gwarp, long long nwarps,
                                           uint4* buf, int lane) {
  long long k = gwarp;
  int head, x;
  if (copy_next_item(j, s, k, nwarps, lane, head, x))
    copy_stage(j, s, head, x, (uint32_t)__cvta_generic_to_shared(buf), lane);
}

__device__ __forceinline__ void copy_finish(const CopyJob& j, const Shape& s, long long gwarp, long long nwarps,
                                            uint4* buf, int lane) {
  long long k = gwarp;
  int head, x;
  bool staged = copy_next_item(j, s, k, nwarps, lane, head, x);
  while (staged) {
    copy_store(j, s, head, x, buf, lane);
    __syncwarp();
    int h2, x2;
    staged = copy_next_item(j, s, k, nwarps, lane, h2, x2);
    if (staged) {
      head = h2;
      x = x2;
      copy_stage(j, s, head, x, (uint32_t)__cvta_generic_to_shared(buf), lane);
    }
  }
}

}  // namespace oasis
