// f3: agreement of a predicted top-K set with the exact one, per (request, KV head).
//
// metalmedia.ai page, Figure 6 caption (per-layer agreement between the top-K
// set the draft query predicts and the exact top-K set of the true next-token
// query) and Figure 4 caption (the same accuracy at K = 20, previous token versus
// lookahead token).  Both sets come from oasis_topk_select, run once with the
// predicting queries and once with the true query as the only lookahead row;
// this kernel only intersects them.
//
// One warp per head: each lane takes every 32nd entry of the exact set and
// binary-searches it in the predicted set (ascending, as oasis_topk_select writes
// it); a hit also counts as attended when the block is resident.  The counts are
// warp sums, so the result does not depend on scheduling.
#include "common.cuh"

namespace oasis {

constexpr int kAgreeWarps = 8;

__global__ void __launch_bounds__(kAgreeWarps * 32)
set_agreement_kernel(Shape s, const int* __restrict__ pred, const int* __restrict__ npred,
                     const int* __restrict__ exact, const int* __restrict__ nexact,
                     const int* __restrict__ blk2slot, int* __restrict__ counts, unsigned* __restrict__ err) {
  const int lane = threadIdx.x & 31;
  const long long head = (long long)blockIdx.x * kAgreeWarps + (threadIdx.x >> 5);
  if (head >= (long long)s.B * s.Hkv) return;
  int na = npred[head], nb = nexact[head];
  unsigned ew = 0;
  if (na < 0 || na > s.Kb) { ew |= OASIS_EW_BAD_COUNT; na = na < 0 ? 0 : s.Kb; }
  if (nb < 0 || nb > s.Kb) { ew |= OASIS_EW_BAD_COUNT; nb = nb < 0 ? 0 : s.Kb; }
  const int* A = pred + head * s.Kb;
  const int* E = exact + head * s.Kb;
  int hit = 0, hit_res = 0;
  for (int i = lane; i < nb; i += 32) {
    const int x = E[i];
    if (x < 0 || x >= s.nb_max) { ew |= OASIS_EW_BAD_BLOCK; continue; }
    int lo = 0, hi = na - 1;
    bool found = false;
    while (lo <= hi) {
      const int mid = (lo + hi) >> 1;
      const int v = A[mid];
      if (v == x) { found = true; break; }
      if (v < x) lo = mid + 1; else hi = mid - 1;
    }
    if (found) {
      ++hit;
      if (blk2slot && blk2slot[head * s.nb_max + x] >= 0) ++hit_res;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    hit += __shfl_xor_sync(0xffffffffu, hit, o);
    hit_res += __shfl_xor_sync(0xffffffffu, hit_res, o);
  }
  if (lane == 0) {
    counts[head * 3 + 0] = hit;
    counts[head * 3 + 1] = blk2slot ? hit_res : -1;
    counts[head * 3 + 2] = nb;
  }
  if (ew && err) atomicOr(err, ew);
}

cudaError_t launch_set_agreement(const Shape& s, const int* pred, const int* npred, const int* exact,
                                 const int* nexact, const int* blk2slot, int* counts, unsigned* err,
                                 cudaStream_t stream) {
  const long long heads = (long long)s.B * s.Hkv;
  const int grid = (int)((heads + kAgreeWarps - 1) / kAgreeWarps);
  set_agreement_kernel<<<grid, kAgreeWarps * 32, 0, stream>>>(s, pred, npred, exact, nexact, blk2slot, counts,
                                                              err);
  return cudaGetLastError();
}

}  // namespace oasis
