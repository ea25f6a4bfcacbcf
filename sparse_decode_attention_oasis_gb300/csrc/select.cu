// a2 top-K under the token budget and a3 capped diff against the resident set.
//
// Both steps pick "the r best candidates by (exact score descending, block index
// ascending)" out of a candidate list: all blocks of a head for the top-K (OasisKV
// abstract: 2,048-token KV budget; Figure 7 caption: top-K blocks), the
// selected-but-missing blocks for the capped fetch list (metalmedia.ai page,
// explanatory figure step 3; Table 2 caption: the per-step fetch cap).
//
// Exact selection from certified intervals.  The scores come with a bound e,
// |s~ - s| <= e.  With t the r-th largest s~, bracketed as t_lo <= t <= t_hi (by
// rank counting, or a histogram pass and rank counting inside the bin that holds
// t), and E = max e over the candidates:
//   s~_i - e_i > t_hi + E  => i is certainly among the r best,
//   s~_i + e_i < t_lo - E  => i certainly is not,
// (every candidate that could rank at or above a "certain" one has s~ > t, and
// at most r-1 do; conversely the r candidates with s~ >= t all rank above a
// "certainly not").  The remaining candidates U are re-scored exactly:
//   1. the block's 16 x N dot products are re-formed on the tensor cores with
//      per-dot bounds 2^-12 |q_n| |k_t| (the scoring kernel's error model, per
//      dot instead of per block), which isolates the dot(s) that can be the
//      block's maximum - normally one;
//   2. those dots are evaluated exactly: each bf16 is m * 2^(E-134), each
//      product is an integer times 2^-266, and a 544-bit two's complement
//      fixed-point number (17 limbs of 32 bits) holds the sum with no rounding
//      (a 64-bit integer warp sum when the products span at most 40 binades,
//      else limb by limb);
//   3. one rank count over U by exact comparison marks its r best (a U larger
//      than Kb is merged into a running top-r set kSelWarps blocks at a time).
// Every routine has one call site per kernel, so that the code a CTA runs once
// stays small: run once per head, the phases are bound by latency, including
// instruction fetch.
// The result equals the definition for every finite input whose tensor-core
// accumulation stays within the modelled bound (the GPU tests check every block
// score of every case against its exact value).
#include "common.cuh"

namespace oasis {

constexpr int kSelThreads = 256;               // threads per CTA (512 for few heads with long contexts)
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kSelMaxWarps = 16;
constexpr int kLimbs = 17;
constexpr int kMaxN = 32;      // lookahead queries x GQA group

struct SelCtx {
  const uint16_t* k;   // keys of this head [T_max][128]
  const uint16_t* q_la;
  int b, h, ctx, N, G, n_la, Hq;
  // shared memory
  uint16_t* qb;                // [kMaxN][128]
  float* qn;                   // [kMaxN]
  uint16_t* kst;               // [kSelWarps][16][128] staged key blocks
  uint32_t* tmp;               // [kSelWarps][kLimbs]
  uint32_t* bval;              // [kSelWarps][kLimbs]
  int* bidx;                   // [kSelWarps]
  uint32_t* tval;              // [Kb][kLimbs] running top-r set (exact values)
  int* tidx;                   // [Kb]
  uint32_t* tval2;             // [Kb][kLimbs] next top-r set
  int* tidx2;                  // [Kb]
  int* rank;                   // [Kb + kSelWarps]
  uint32_t* hist;              // [256]
  int* scal;                   // [8] scalars
  float* fscal;                // [kSelWarps]
  int qstate;                  // queries: 0 not staged, 1 copies in flight, 3 landed (visible after the
                               // next CTA barrier), 2 staged with norms
  int kcap;                    // entries of tval (Kb)
};

__device__ __forceinline__ void sel_cp_async16(void* dst, const void* src) {
  const uint32_t d = (uint32_t)__cvta_generic_to_shared(dst);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(src) : "memory");
}
__device__ __forceinline__ void sel_cp_async_wait_all() {
  asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

// ---------------------------------------------------------------- exact arithmetic
// Sign of a - b for two 544-bit two's complement numbers (kLimbs words, least
// significant first).  Every limb is loaded and compared at once; a higher
// differing limb overrides a lower one, the top limb compares signed.
__device__ __forceinline__ int exact_cmp(const uint32_t* a, const uint32_t* b) {
  int r = 0;
#pragma unroll
  for (int i = 0; i < kLimbs - 1; ++i) {
    const uint32_t x = a[i], y = b[i];
    r = x != y ? (x < y ? -1 : 1) : r;
  }
  const int ta = (int)a[kLimbs - 1], tb = (int)b[kLimbs - 1];
  return ta != tb ? (ta < tb ? -1 : 1) : r;
}

// Exact product of one bf16 pair as mms * 2^(ee - 266): mms the signed product of
// the two 8-bit significands (|mms| < 2^16), ee in 0 .. 508 (mms = 0: no term).
__device__ __forceinline__ void exact_prod(uint32_t qb, uint32_t kb, long long& mms, int& ee) {
  const uint32_t kE = (kb >> 7) & 0xffu, qE = (qb >> 7) & 0xffu;
  const uint32_t km = (kb & 0x7fu) | (kE ? 0x80u : 0u);
  const uint32_t qm = (qb & 0x7fu) | (qE ? 0x80u : 0u);
  const uint32_t mm = km * qm;
  ee = (int)(kE ? kE : 1u) + (int)(qE ? qE : 1u) - 2;
  mms = ((kb ^ qb) & 0x8000u) ? -(long long)mm : (long long)mm;
}

// The general case of warp_exact_dot (products spread over more than 40 binades;
// rare, so kept out of line): each lane forms its products as (limb, low 32
// bits, high bits); the limbs the warp touches are summed one at a time with a
// 64-bit warp reduction (no atomics), then every lane runs the same carry chain
// and lane i < 17 stores limb i.
template <bool kBox>
__device__ __noinline__ void warp_exact_dot_limbs(const uint16_t* krow, const uint16_t* qrow, uint32_t* out, int lane,
                                                  const uint16_t* krow_neg) {
  int limb[4];
  long long lo[4], hi[4];
  int lmin = kLimbs, lmax = -1;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int e = lane + 32 * j;
    const uint32_t qb = qrow[e];
    const uint32_t kb = (kBox && (qb & 0x8000u)) ? krow_neg[e] : krow[e];
    long long mms;
    int ee;
    exact_prod(qb, kb, mms, ee);
    limb[j] = -2;
    lo[j] = hi[j] = 0;
    if (mms) {
      const unsigned long long v = (unsigned long long)(mms < 0 ? -mms : mms) << (ee & 31);
      lo[j] = (long long)(v & 0xffffffffull);
      hi[j] = (long long)(v >> 32);
      if (mms < 0) {
        lo[j] = -lo[j];
        hi[j] = -hi[j];
      }
      limb[j] = ee >> 5;
      lmin = min(lmin, limb[j]);
      lmax = max(lmax, limb[j] + 1);
    }
  }
  lmin = __reduce_min_sync(0xffffffffu, lmin);
  lmax = __reduce_max_sync(0xffffffffu, lmax);
  long long mine = 0;
  for (int L = lmin; L <= lmax; ++L) {
    long long sum = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (limb[j] == L) sum += lo[j];
      if (limb[j] + 1 == L) sum += hi[j];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    if (lane == L) mine = sum;
  }
  long long carry = 0;
  uint32_t word = 0;
  for (int i = 0; i < kLimbs; ++i) {
    const long long v = __shfl_sync(0xffffffffu, mine, i) + carry;
    if (lane == i) word = (uint32_t)(unsigned long long)v;
    carry = v >> 32;
  }
  if (lane < kLimbs) out[lane] = word;
  __syncwarp();
}

// Exact q.k (times 2^266) of a 128-long bf16 row pair, by one warp, as kLimbs
// words.  Each product is mm * 2^(ee - 266) with |mm| < 2^16.  When the nonzero
// products' ee span at most 40 (the usual case), sum_j mm_j 2^(ee_j - emin) over
// 128 products is below 2^63 and is summed exactly in 64-bit integers; lane i
// then writes limb i of that sum shifted by emin.  Otherwise warp_exact_dot_limbs
// sums it limb by limb.  With kBox the key element is chosen per dimension by the
// query's sign: krow (the pooled maxima) where q >= 0, krow_neg (the minima) where
// q < 0, which makes the sum the pooled score sum_i max(q_i hi_i, q_i lo_i).
template <bool kBox>
__device__ __forceinline__ void warp_exact_dot(const uint16_t* krow, const uint16_t* qrow, uint32_t* out, int lane,
                                               const uint16_t* krow_neg = nullptr) {
  long long mms[4];
  int eev[4];
  int emin = 1 << 20, emax = -1;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int e = lane + 32 * j;
    const uint32_t qb = qrow[e];
    const uint32_t kb = (kBox && (qb & 0x8000u)) ? krow_neg[e] : krow[e];
    exact_prod(qb, kb, mms[j], eev[j]);
    if (mms[j]) {
      emin = min(emin, eev[j]);
      emax = max(emax, eev[j]);
    }
  }
  emin = __reduce_min_sync(0xffffffffu, emin);
  emax = __reduce_max_sync(0xffffffffu, emax);
  if (emax >= 0 && emax - emin > 40) {
    warp_exact_dot_limbs<kBox>(krow, qrow, out, lane, krow_neg);
    return;
  }
  long long acc = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j)
    if (mms[j]) acc += mms[j] * (1LL << (eev[j] - emin));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  // limb i of |acc| * 2^emin, then two's complement if negative: the +1 carries
  // into limb i exactly when every lower limb of the magnitude is zero
  const unsigned long long mag = acc < 0 ? (unsigned long long)(-acc) : (unsigned long long)acc;
  uint32_t w = 0u;
  if (emax >= 0 && lane < kLimbs) {
    const int b = 32 * lane - emin;  // bit of mag that lands at bit 0 of limb `lane`
    if (b >= 0 && b < 64) w = (uint32_t)(mag >> b);
    else if (b < 0 && b > -32) w = (uint32_t)(mag << (-b));
  }
  const unsigned nz = __ballot_sync(0xffffffffu, w != 0u);
  if (acc < 0) {
    const uint32_t carry = (nz & ((1u << lane) - 1u)) == 0u ? 1u : 0u;
    w = ~w + carry;
  }
  if (lane < kLimbs) out[lane] = w;
  __syncwarp();
}

// ---------------------------------------------------------------- block-wide helpers
__device__ __forceinline__ int block_excl_scan(int v, int* red, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) red[warp] = x;
  __syncthreads();
  const int nw = blockDim.x >> 5;
  if (warp == 0) {
    int w = lane < nw ? red[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < nw) red[lane] = w;
    if (lane == nw - 1) *total = w;
  }
  __syncthreads();
  const int base = warp ? red[warp - 1] : 0;
  const int res = base + x - v;
  __syncthreads();
  return res;
}

__device__ __forceinline__ float block_max(float v, float* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = warp_max(v);
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float r = red[0];
  for (int i = 1; i < (int)(blockDim.x >> 5); ++i) r = fmaxf(r, red[i]);
  __syncthreads();
  return r;
}

// Lists up to this long get their k-th largest by rank counting.
constexpr int kRankMax = kSelThreads;

// The k-th largest (1 <= k <= m) of v[0], v[kStride], ..., v[(m-1) kStride]: the
// value with fewer than k larger values and at least k values at least as large
// (thread i takes values i, i + blockDim.x, ...; every thread that finds it writes
// the same value to *out).  Ends with *out visible to the CTA.
template <int kStride>
__device__ void kth_by_rank(const float* v, int m, int k, float* out) {
  for (int i = threadIdx.x; i < m; i += blockDim.x) {
    const float x = v[i * kStride];
    int gt = 0, ge = 0;
#pragma unroll 8
    for (int j = 0; j < m; ++j) {
      const float y = v[j * kStride];
      gt += y > x ? 1 : 0;
      ge += y >= x ? 1 : 0;
    }
    if (gt < k && k <= ge) *out = x;
  }
  __syncthreads();
}

// Small k (the per-step fetch cap): the k-th largest of se[0..n).x, n <= 256, by
// one warp: each lane holds up to 8 values; every round takes the warp's largest
// remaining value and counts its copies, until k values have been counted.
constexpr int kSmallK = 16;
__device__ void kth_small_k(const float2* se, int n, int k, float* out) {
  const int lane = threadIdx.x & 31;
  float v[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) v[j] = lane + 32 * j < n ? se[lane + 32 * j].x : neg_inf();
  int left = k;
  for (int round = 0; round < k; ++round) {
    float m = v[0];
#pragma unroll
    for (int j = 1; j < 8; ++j) m = fmaxf(m, v[j]);
    m = warp_max(m);
    int cnt = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) cnt += __popc(__ballot_sync(0xffffffffu, v[j] == m));
    if (cnt >= left) {
      if (lane == 0) *out = m;
      return;
    }
    left -= cnt;
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = v[j] == m ? neg_inf() : v[j];
  }
}

// Bracket [t_lo, t_hi] around the k-th largest s~ among se[0..n) (1 <= k <= n), and
// E = max e.  Up to kRankMax entries: t itself, by rank counting.  Longer lists:
// a pass of 256 bins, bin1 = floor(256 (x - min)/(max - min)), finds the bin that
// holds the k-th largest; if that bin holds at most kRankMax entries they are
// listed (in `scratch`, n floats) and t is found among them by rank counting,
// otherwise a second pass of 256 sub-bins of bin1's fraction narrows it to the
// cell's smallest and largest s~.  Both bin maps are monotone in x (one
// subtraction and a multiplication by a positive constant, exact sub-bin
// offsets), so the k-th largest lies in the selected bin and cell.
__device__ void kth_bracket(const float2* se, int n, int k, uint32_t* hist, int* scal, float* fs, float* scratch,
                            uint8_t* bins, float& t_lo, float& t_hi, float& emax) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float* tslot = fs + 60;   // fs[0 .. 3 kSelWarps) hold the partial reductions, fs + 64 the cell keys
  float mn = __int_as_float(0x7f800000), mx = neg_inf(), em = 0.f;
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    const float2 v = se[i];
    mn = fminf(mn, v.x);
    mx = fmaxf(mx, v.x);
    em = fmaxf(em, v.y);
  }
  mn = -warp_max(-mn);
  mx = warp_max(mx);
  em = warp_max(em);
  if (lane == 0) { fs[3 * warp] = mn; fs[3 * warp + 1] = mx; fs[3 * warp + 2] = em; }
  const bool small = n <= kRankMax;
  if (!small)
    for (int i = threadIdx.x; i < 256; i += blockDim.x) hist[i] = 0u;
  if (threadIdx.x == 0) { *tslot = neg_inf(); scal[5] = 0; }
  __syncthreads();
  mn = fs[0]; mx = fs[1]; em = fs[2];
  for (int w = 1; w < (int)(blockDim.x >> 5); ++w) {
    mn = fminf(mn, fs[3 * w]); mx = fmaxf(mx, fs[3 * w + 1]); em = fmaxf(em, fs[3 * w + 2]);
  }
  emax = em;
  if (small) {
    if (k <= kSmallK) {
      if (warp == 0) kth_small_k(se, n, k, tslot);
      __syncthreads();
    } else {
      kth_by_rank<2>(reinterpret_cast<const float*>(se), n, k, tslot);
    }
    t_lo = t_hi = *tslot;
    __syncthreads();
    return;
  }
  const float span = mx - mn;
  const float sc1 = span > 1e-30f ? 256.0f / span : 0.f;
  // pass 1: plain shared-memory atomics (a warp's same-bin lanes serialise in
  // hardware, far cheaper than grouping them first); each entry's bin is kept
  // in `bins` for the listing pass
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    const int bin = min(255, (int)((se[i].x - mn) * sc1));
    bins[i] = (uint8_t)bin;
    atomicAdd(&hist[bin], 1u);
  }
  __syncthreads();
  if (warp == 0) {
    uint32_t c[8], sum = 0;
#pragma unroll
    for (int q = 0; q < 8; ++q) { c[q] = hist[255 - (lane * 8 + q)]; sum += c[q]; }
    uint32_t incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    const uint32_t excl = incl - sum;
    if (excl < (uint32_t)k && (uint32_t)k <= incl) {
      uint32_t run = excl;
      for (int q = 0; q < 8; ++q) {
        if (run + c[q] >= (uint32_t)k) { scal[0] = 255 - (lane * 8 + q); scal[1] = (int)run; break; }
        run += c[q];
      }
    }
  }
  __syncthreads();
  const int b1 = scal[0];
  const int k1 = k - scal[1];
  const int m1 = (int)hist[b1];
  if (m1 <= kRankMax) {
    // list bin b1's entries (a handful: one shared atomic each), then rank them
    for (int i = threadIdx.x; i < n; i += blockDim.x)
      if (bins[i] == (uint8_t)b1) scratch[atomicAdd(&scal[5], 1)] = se[i].x;
    __syncthreads();
    kth_by_rank<1>(scratch, m1, k1, tslot);
    t_lo = t_hi = *tslot;
    __syncthreads();
    return;
  }
  uint32_t* h2 = hist + 256;                    // reuse: counts of sub-bins
  uint32_t* kmin = reinterpret_cast<uint32_t*>(fs + 64);   // per sub-bin min / max keys
  uint32_t* kmax = kmin + 256;
  for (int i = threadIdx.x; i < 256; i += blockDim.x) { h2[i] = 0u; kmin[i] = 0xffffffffu; kmax[i] = 0u; }
  __syncthreads();
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    if (bins[i] != (uint8_t)b1) continue;
    const float x = se[i].x;
    const float y = (x - mn) * sc1;
    const int bb1 = min(255, (int)y);  // == b1: the same arithmetic as pass 1
    const uint32_t bin = (uint32_t)max(0, min(255, (int)((y - (float)bb1) * 256.0f)));
    const uint32_t key = float_key(x);
    atomicMin(&kmin[bin], key);
    atomicMax(&kmax[bin], key);
    atomicAdd(&h2[bin], 1u);
  }
  __syncthreads();
  if (warp == 0) {
    uint32_t c[8], sum = 0;
#pragma unroll
    for (int q = 0; q < 8; ++q) { c[q] = h2[255 - (lane * 8 + q)]; sum += c[q]; }
    uint32_t incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    const uint32_t excl = incl - sum;
    if (excl < (uint32_t)k1 && (uint32_t)k1 <= incl) {
      uint32_t run = excl;
      for (int q = 0; q < 8; ++q) {
        if (run + c[q] >= (uint32_t)k1) { scal[2] = 255 - (lane * 8 + q); break; }
        run += c[q];
      }
    }
  }
  __syncthreads();
  t_lo = key_float(kmin[scal[2]]);
  t_hi = key_float(kmax[scal[2]]);
  __syncthreads();
}

// Start copying the head's lookahead queries (bf16 bits) into shared memory with
// 16-byte cp.async, so that their latency overlaps the bracket and classification.
__device__ void issue_queries(SelCtx& c) {
  for (int idx = threadIdx.x; idx < c.N * 16; idx += blockDim.x) {
    const int n = idx >> 4, part = idx & 15;
    const int j = n / c.G, gg = n - j * c.G;
    sel_cp_async16(c.qb + n * kD + part * 8,
                   c.q_la + (((long long)c.b * c.n_la + j) * c.Hq + c.h * c.G + gg) * kD + part * 8);
  }
  c.qstate = 1;
}

// Make the head's lookahead queries (bf16 bits and fp32 norms) ready in shared
// memory: finish the copies issue_queries started, or load them now (one 16-byte
// load per piece, all issued together).  Idempotent; every thread calls it.
__device__ void stage_queries(SelCtx& c) {
  if (c.qstate == 2) return;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (c.qstate == 3) {
    // landed and visible already (a CTA barrier followed every thread's wait)
  } else if (c.qstate == 1) {
    sel_cp_async_wait_all();
  } else {
    for (int idx = threadIdx.x; idx < c.N * 16; idx += blockDim.x) {
      const int n = idx >> 4, part = idx & 15;
      const int j = n / c.G, gg = n - j * c.G;
      const uint4 v = ldg_nc(c.q_la + (((long long)c.b * c.n_la + j) * c.Hq + c.h * c.G + gg) * kD + part * 8);
      reinterpret_cast<uint4*>(c.qb + n * kD)[part] = v;
    }
  }
  if (c.qstate != 3) __syncthreads();  // state 3: already visible
  for (int n = warp; n < c.N; n += (int)(blockDim.x >> 5)) {
    const uint32_t w0 = reinterpret_cast<const uint32_t*>(c.qb + n * kD)[lane];
    const uint32_t w1 = reinterpret_cast<const uint32_t*>(c.qb + n * kD)[lane + 32];
    float ss = bf_lo(w0) * bf_lo(w0);
    ss = fmaf(bf_hi(w0), bf_hi(w0), ss);
    ss = fmaf(bf_lo(w1), bf_lo(w1), ss);
    ss = fmaf(bf_hi(w1), bf_hi(w1), ss);
    ss = warp_sum(ss);
    if (lane == 0) c.qn[n] = sqrtf(ss);
  }
  __syncthreads();
  c.qstate = 2;
}

__device__ __forceinline__ uint4 lds16v(const uint16_t* p) { return *reinterpret_cast<const uint4*>(p); }

// Exact score (x 2^266, as kLimbs words) of block `blk`, by one warp, into out.
// The block's 16 key rows (4 KiB) are staged in this warp's shared-memory slot with
// one round of coalesced 16-byte loads.  The 16 x N dot products are then formed
// on the tensor cores exactly as the scoring kernel forms them (bf16 in, fp32
// accumulate, so the same bound 2^-12 |q_n| |k_t| holds for each dot); only the
// dots whose interval reaches the best lower bound of the block are summed
// exactly.  Usually that is one dot.
__device__ void warp_exact_block_score(const SelCtx& c, int blk, uint32_t* out, int warp, int lane) {
  const int g = lane >> 2, t = lane & 3;
  uint16_t* kst = c.kst + warp * (kBS * kD);
  {
    const uint4* src = reinterpret_cast<const uint4*>(c.k + (long long)blk * kBS * kD);
    uint4* dst = reinterpret_cast<uint4*>(kst);
    uint4 v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = ldg_nc(src + lane + 32 * i);
#pragma unroll
    for (int i = 0; i < 8; ++i) dst[lane + 32 * i] = v[i];
  }
  __syncwarp();
  uint4 ra[4], rb[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    ra[i] = lds16v(kst + g * kD + (t + 4 * i) * 8);
    rb[i] = lds16v(kst + (g + 8) * kD + (t + 4 * i) * 8);
  }
  // token norms of rows g and g+8
  float s0 = 0.f, s1 = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t A[4] = {ra[i].x, ra[i].y, ra[i].z, ra[i].w};
    const uint32_t Bw[4] = {rb[i].x, rb[i].y, rb[i].z, rb[i].w};
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      s0 = fmaf(bf_lo(A[m]), bf_lo(A[m]), s0); s0 = fmaf(bf_hi(A[m]), bf_hi(A[m]), s0);
      s1 = fmaf(bf_lo(Bw[m]), bf_lo(Bw[m]), s1); s1 = fmaf(bf_hi(Bw[m]), bf_hi(Bw[m]), s1);
    }
  }
  s0 += __shfl_xor_sync(0xffffffffu, s0, 1);
  s0 += __shfl_xor_sync(0xffffffffu, s0, 2);
  s1 += __shfl_xor_sync(0xffffffffu, s1, 1);
  s1 += __shfl_xor_sync(0xffffffffu, s1, 2);
  const float kn0 = sqrtf(s0), kn1 = sqrtf(s1);
  const int NT = (c.N + 7) >> 3;
  float acc[4][4];
#pragma unroll
  for (int nt = 0; nt < 4; ++nt) {
    acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
    if (nt < NT) {
      const int n = nt * 8 + g;
      uint4 qv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
        qv[i] = n < c.N ? lds16v(c.qb + n * kD + (t + 4 * i) * 8) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t A[4] = {ra[i].x, ra[i].y, ra[i].z, ra[i].w};
        const uint32_t Bw[4] = {rb[i].x, rb[i].y, rb[i].z, rb[i].w};
        const uint32_t Q[4] = {qv[i].x, qv[i].y, qv[i].z, qv[i].w};
#pragma unroll
        for (int hh = 0; hh < 2; ++hh)
          mma_bf16_16816(acc[nt][0], acc[nt][1], acc[nt][2], acc[nt][3], A[2 * hh], Bw[2 * hh], A[2 * hh + 1],
                         Bw[2 * hh + 1], Q[2 * hh], Q[2 * hh + 1]);
      }
    }
  }
  // per-dot intervals; element e of n-tile nt is (token g or g+8, query nt*8 + 2t + (e & 1))
  const int tok0 = blk * kBS + g;
  float vlo[16], vhi[16];
  float best_lo = neg_inf();
#pragma unroll
  for (int nt = 0; nt < 4; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int n = nt * 8 + 2 * t + (e & 1);
      const bool row8 = e >= 2;
      const bool ok = nt < NT && n < c.N && (tok0 + (row8 ? 8 : 0)) < c.ctx;
      const int idx = nt * 4 + e;
      vlo[idx] = neg_inf();
      vhi[idx] = neg_inf();
      if (ok) {
        const float v = acc[nt][e];
        const float eps = __fmaf_ru(kAccRel * 1.0009765625f, __fmul_ru(row8 ? kn1 : kn0, c.qn[n]),
                                    7.52316384526264e-37f /* 2^-120 */);
        vlo[idx] = __fsub_rd(v, eps);
        vhi[idx] = __fadd_ru(v, eps);
        if (!(fabsf(v) <= 3.0e38f)) { vlo[idx] = neg_inf(); vhi[idx] = __int_as_float(0x7f800000); }
        best_lo = fmaxf(best_lo, vlo[idx]);
      }
    }
  best_lo = warp_max(best_lo);
  // bit idx of `mine`: this lane's dot idx can be the block's maximum
  unsigned mine = 0u;
#pragma unroll
  for (int idx = 0; idx < 16; ++idx)
    if (vhi[idx] != neg_inf() && vhi[idx] >= best_lo) mine |= 1u << idx;
  bool have = false;
  uint32_t* tmp = c.tmp + warp * kLimbs;
  // one candidate dot at a time (lowest lane first, then lowest idx), summed exactly
  for (unsigned lanes = __ballot_sync(0xffffffffu, mine != 0u); lanes;
       lanes = __ballot_sync(0xffffffffu, mine != 0u)) {
    const int src = __ffs(lanes) - 1;
    const int idx = __ffs(__shfl_sync(0xffffffffu, mine, src)) - 1;
    if (lane == src) mine &= mine - 1u;
    const int sg = src >> 2, st = src & 3;
    const int nt = idx >> 2, e = idx & 3;
    const int tau = sg + (e >= 2 ? 8 : 0);
    const int n = nt * 8 + 2 * st + (e & 1);
    warp_exact_dot<false>(kst + tau * kD, c.qb + n * kD, tmp, lane);
    if (lane == 0) {
      if (!have || exact_cmp(tmp, out) > 0)
        for (int i = 0; i < kLimbs; ++i) out[i] = tmp[i];
    }
    have = true;
    __syncwarp();
  }
  if (!have && lane == 0) {
    for (int i = 0; i < kLimbs - 1; ++i) out[i] = 0u;
    out[kLimbs - 1] = 0x80000000u;
  }
  __syncwarp();
}

// Exact pooled score (x 2^266) of block `blk` (f1: max over the queries n of
// sum_i max(q_ni hi_i, q_ni lo_i)), by one warp, into out.  The block's two pooled
// rows (512 bytes) are staged in the warp's slot; each query's sum is first formed
// in fp32 from its exact products (4 per lane, then a 5-level tree) with the bound
// 2^-16 sum|p| + 2^-120 (at most 8 roundings of 2^-24 of that sum, plus
// underflowed products); only the queries whose interval reaches the best lower
// bound are summed exactly.
__device__ void warp_exact_pooled_score(const SelCtx& c, int blk, uint32_t* out, int warp, int lane) {
  uint16_t* kst = c.kst + warp * (kBS * kD);
  reinterpret_cast<uint4*>(kst)[lane] = ldg_nc(reinterpret_cast<const uint4*>(c.k + (long long)blk * 2 * kD) + lane);
  __syncwarp();
  const uint16_t* hi = kst;
  const uint16_t* lo = kst + kD;
  // Screening: fp32 pooled dots with error bounds, P lanes per query (the largest
  // power of two with N * P <= 32), each over 128 / P elements taken as bf16 pairs,
  // then log2(P) shuffles.  Lane rotation of the word index keeps the shared-memory
  // reads of one instruction in distinct banks.  Any summation order of the 128
  // exact products errs by at most 127 * 2^-24 < 2^-16 of their absolute sum.
  int P = 1;
  while (c.N * P * 2 <= 32) P *= 2;
  const int n = lane / P, part = lane - n * P;
  const int wpl = 64 / P;  // bf16 pairs per lane
  float v0 = 0.f, v1 = 0.f, a0 = 0.f, a1 = 0.f;
  if (n < c.N) {
    const uint32_t* qw = reinterpret_cast<const uint32_t*>(c.qb + n * kD) + part * wpl;
    const uint32_t* hw = reinterpret_cast<const uint32_t*>(hi) + part * wpl;
    const uint32_t* lw = reinterpret_cast<const uint32_t*>(lo) + part * wpl;
    for (int w = 0; w < wpl; ++w) {
      const int ww = (w + lane) & (wpl - 1);
      const uint32_t qv = qw[ww], hv = hw[ww], lv = lw[ww];
      // a negative query element meets the block's minimum, a non-negative one its maximum
      const float p0 = bf_lo(qv) * ((qv & 0x8000u) ? bf_lo(lv) : bf_lo(hv));
      const float p1 = bf_hi(qv) * ((qv & 0x80000000u) ? bf_hi(lv) : bf_hi(hv));
      v0 += p0;
      a0 += fabsf(p0);
      v1 += p1;
      a1 += fabsf(p1);
    }
  }
  float v = v0 + v1, a = a0 + a1;
  for (int o = 1; o < P; o <<= 1) {
    v += __shfl_xor_sync(0xffffffffu, v, o);
    a += __shfl_xor_sync(0xffffffffu, a, o);
  }
  float my_lo = neg_inf(), my_hi = neg_inf();
  if (part == 0 && n < c.N) {
    const float eps = __fmaf_ru(1.52587890625e-05f /* 2^-16 */, a, 7.52316384526264e-37f /* 2^-120 */);
    my_lo = __fsub_rd(v, eps);
    my_hi = __fadd_ru(v, eps);
    if (!(fabsf(v) <= 3.0e38f) || !(a <= 3.0e38f)) { my_lo = neg_inf(); my_hi = __int_as_float(0x7f800000); }
  }
  const float best_lo = warp_max(my_lo);
  unsigned mask = __ballot_sync(0xffffffffu, part == 0 && n < c.N && my_hi >= best_lo);
  uint32_t* tmp = c.tmp + warp * kLimbs;
  bool have = false;
  while (mask) {
    const int qn = (__ffs(mask) - 1) / P;
    mask &= mask - 1;
    warp_exact_dot<true>(hi, c.qb + qn * kD, tmp, lane, lo);
    if (lane == 0) {
      if (!have || exact_cmp(tmp, out) > 0)
        for (int i = 0; i < kLimbs; ++i) out[i] = tmp[i];
    }
    have = true;
    __syncwarp();
  }
  if (!have && lane == 0) {
    for (int i = 0; i < kLimbs - 1; ++i) out[i] = 0u;
    out[kLimbs - 1] = 0x80000000u;
  }
  __syncwarp();
}

// Mark (cls = 1) the r best of the uncertain candidates U[0..nU) by exact order;
// cand_blk maps a candidate index to its block (nullptr = identity).  Up to Kb
// candidates: every warp scores candidates warp, warp + kSelWarps, ... into tval,
// then each candidate's rank is the number of candidates ordered before it (exact
// value descending, block ascending) and the r first are marked.  More than Kb
// (rare; bounded memory): the running top-r set T (exact values, in rank order)
// is merged with each batch of kSelWarps freshly scored blocks by counting, for
// every member of the union, how many members rank before it; the r first go to
// the other buffer.
template <bool kPooled>
__device__ void refine_top_r(SelCtx& c, const int* U, int nU, int r, const int* cand_blk,
                             uint8_t* cls) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  stage_queries(c);
  const bool single = nU <= c.kcap;
  const int nw = blockDim.x >> 5;
  const int chunk = single ? nU : nw;
  uint32_t* vals = single ? c.tval : c.bval;  // exact values of this round's candidates
  int tcount = 0;
  uint32_t* tv = c.tval;
  int* ti = c.tidx;
  uint32_t* tv2 = c.tval2;
  int* ti2 = c.tidx2;
  for (int base = 0; base < nU; base += chunk) {
    const int nbat = min(chunk, nU - base);
    for (int i = warp; i < nbat; i += nw) {
      const int ci = U[base + i];
      const int blk = cand_blk ? cand_blk[ci] : ci;
      if constexpr (kPooled)
        warp_exact_pooled_score(c, blk, vals + i * kLimbs, warp, lane);
      else
        warp_exact_block_score(c, blk, vals + i * kLimbs, warp, lane);
      if (lane == 0 && !single) c.bidx[i] = ci;
    }
    __syncthreads();
    if (single) {
      for (int m = threadIdx.x; m < nU; m += blockDim.x) {
        uint32_t mv[kLimbs];
#pragma unroll
        for (int i = 0; i < kLimbs; ++i) mv[i] = vals[m * kLimbs + i];
        const int mci = U[m];
        const int mblk = cand_blk ? cand_blk[mci] : mci;
        int rk = 0;
        for (int o = 0; o < nU; ++o) {
          const int oci = U[o];
          const int oblk = cand_blk ? cand_blk[oci] : oci;
          const int cmpv = exact_cmp(vals + o * kLimbs, mv);
          rk += (cmpv > 0 || (cmpv == 0 && oblk < mblk)) ? 1 : 0;
        }
        cls[mci] = rk < r ? 1 : 0;
      }
      __syncthreads();
      return;
    }
    const int tot = tcount + nbat;
    for (int m = threadIdx.x; m < tot; m += blockDim.x) {
      const uint32_t* mv = m < tcount ? tv + m * kLimbs : c.bval + (m - tcount) * kLimbs;
      const int midx = m < tcount ? ti[m] : c.bidx[m - tcount];
      const int mblk = cand_blk ? cand_blk[midx] : midx;
      int rk = 0;
      for (int o = 0; o < tot; ++o) {
        if (o == m) continue;
        const uint32_t* ov = o < tcount ? tv + o * kLimbs : c.bval + (o - tcount) * kLimbs;
        const int oidx = o < tcount ? ti[o] : c.bidx[o - tcount];
        const int oblk = cand_blk ? cand_blk[oidx] : oidx;
        const int cmpv = exact_cmp(ov, mv);
        if (cmpv > 0 || (cmpv == 0 && oblk < mblk)) ++rk;
      }
      c.rank[m] = rk;
    }
    __syncthreads();
    for (int m = threadIdx.x; m < tot; m += blockDim.x) {
      const int rk = c.rank[m];
      if (rk >= r) continue;
      const uint32_t* mv = m < tcount ? tv + m * kLimbs : c.bval + (m - tcount) * kLimbs;
#pragma unroll
      for (int i = 0; i < kLimbs; ++i) tv2[rk * kLimbs + i] = mv[i];
      ti2[rk] = m < tcount ? ti[m] : c.bidx[m - tcount];
    }
    tcount = min(r, tot);
    __syncthreads();
    uint32_t* sv = tv; tv = tv2; tv2 = sv;
    int* si = ti; ti = ti2; ti2 = si;
  }
  for (int i = threadIdx.x; i < nU; i += blockDim.x) cls[U[i]] = 0;
  __syncthreads();
  for (int i = threadIdx.x; i < tcount; i += blockDim.x) cls[ti[i]] = 1;
  __syncthreads();
}

// cls[i] = 1 for the k best of the n candidates (exact order), 0 otherwise.
template <bool kPooled>
__device__ void select_best(SelCtx& c, const float2* se, int n, int k, const int* cand_blk,
                            uint8_t* cls, int* U) {
  if (k >= n || k <= 0) {
    for (int i = threadIdx.x; i < n; i += blockDim.x) cls[i] = k > 0 ? 1 : 0;
    __syncthreads();
    return;
  }
  float t_lo, t_hi, em;
  kth_bracket(se, n, k, c.hist, c.scal, c.fscal, reinterpret_cast<float*>(U), cls, t_lo, t_hi, em);
  const float hi_t = __fadd_ru(t_hi, em), lo_t = __fsub_rd(t_lo, em);
  if (threadIdx.x == 0) { c.scal[2] = 0; c.scal[3] = 0; }
  // the queries copied at kernel start have landed once every thread has waited
  // for its own copies; the barrier below makes them visible to the whole CTA
  if (c.qstate == 1) {
    sel_cp_async_wait_all();
    c.qstate = 3;
  }
  __syncthreads();
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    const float2 v = se[i];
    const float lo = __fsub_rd(v.x, v.y), hi = __fadd_ru(v.x, v.y);
    uint8_t cl;
    if (lo > hi_t) {
      cl = 1;
      atomicAdd(&c.scal[3], 1);
    } else if (hi < lo_t) {
      cl = 0;
    } else {
      cl = 2;
      U[atomicAdd(&c.scal[2], 1)] = i;
    }
    cls[i] = cl;
  }
  __syncthreads();
  const int nU = c.scal[2], nin = c.scal[3];
  __syncthreads();
  const int r = k - nin;
  if (r <= 0 || r >= nU) {
    for (int i = threadIdx.x; i < nU; i += blockDim.x) cls[U[i]] = r > 0 ? 1 : 0;
    __syncthreads();
    return;
  }
  // the refine takes one block per warp and round: bring the keys of the later
  // rounds (up to kPrefetchBlocks blocks) into L2 now
  constexpr int kLines = kPooled ? 2 * kD * 2 / 128 : kBS * kD * 2 / 128;
  constexpr int kPrefetchBlocks = 64;
  const int nw = blockDim.x >> 5;
  const int npre = min(nU, nw + kPrefetchBlocks) - nw;
  for (int idx = threadIdx.x; idx < npre * kLines; idx += blockDim.x) {
    const int ci = U[nw + idx / kLines];
    const int blk = cand_blk ? cand_blk[ci] : ci;
    const char* line = reinterpret_cast<const char*>(c.k + (long long)blk * (kPooled ? 2 * kD : kBS * kD)) +
                       (idx % kLines) * 128;
    asm volatile("prefetch.global.L2 [%0];" ::"l"(line));
  }
  refine_top_r<kPooled>(c, U, nU, r, cand_blk, cls);
}

// ---------------------------------------------------------------- shared memory layout
struct SelLayout {
  size_t se, cls, U, cblk, kst, qb, qn, tmp, bval, bidx, tval, tidx, tval2, tidx2, rank, hist, scal,
      fscal, red, total;
};

__host__ __device__ inline size_t align16(size_t x) { return (x + 15) & ~size_t(15); }

// ncap: entries of the candidate list; kb: the budget (the diff's lists are at most
// kb long); nw: warps per CTA.
__host__ __device__ inline SelLayout sel_layout(int ncap, bool with_cblk, int kb, int nw = kSelWarps) {
  SelLayout L;
  size_t o = 0;
  L.se = o; o = align16(o + sizeof(float2) * ncap);
  L.cls = o; o = align16(o + ncap);
  L.U = o; o = align16(o + sizeof(int) * ncap);
  L.cblk = o; o = align16(o + (with_cblk ? sizeof(int) * kb : 0));
  L.kst = o; o = align16(o + sizeof(uint16_t) * nw * kBS * kD);
  L.qb = o; o = align16(o + sizeof(uint16_t) * kMaxN * kD);
  L.qn = o; o = align16(o + sizeof(float) * kMaxN);
  L.tmp = o; o = align16(o + sizeof(uint32_t) * nw * kLimbs);
  L.bval = o; o = align16(o + sizeof(uint32_t) * nw * kLimbs);
  L.bidx = o; o = align16(o + sizeof(int) * nw);
  L.tval = o; o = align16(o + sizeof(uint32_t) * kb * kLimbs);
  L.tidx = o; o = align16(o + sizeof(int) * kb);
  L.tval2 = o; o = align16(o + sizeof(uint32_t) * kb * kLimbs);
  L.tidx2 = o; o = align16(o + sizeof(int) * kb);
  L.rank = o; o = align16(o + sizeof(int) * (kb + nw));
  L.hist = o; o = align16(o + sizeof(uint32_t) * 512);
  L.scal = o; o = align16(o + sizeof(int) * 8);
  L.fscal = o; o = align16(o + sizeof(float) * (64 + 512));
  L.red = o; o = align16(o + sizeof(int) * 32);
  L.total = o;
  return L;
}

// keys: the full keys [heads][nb_max*16][128], or with `pooled` the pooled keys
// [heads][nb_max][2][128].
__device__ SelCtx make_ctx(char* sm, const SelLayout& L, const Shape& s, const uint16_t* keys,
                           const uint16_t* q_la, int head, int ctx, bool pooled) {
  SelCtx c;
  c.b = head / s.Hkv;
  c.h = head - c.b * s.Hkv;
  c.k = keys + (long long)head * s.nb_max * (pooled ? 2 * kD : kBS * kD);
  c.q_la = q_la;
  c.ctx = ctx;
  c.G = s.Hq / s.Hkv;
  c.N = s.n_la * c.G;
  c.n_la = s.n_la;
  c.Hq = s.Hq;
  c.qb = reinterpret_cast<uint16_t*>(sm + L.qb);
  c.qn = reinterpret_cast<float*>(sm + L.qn);
  c.kst = reinterpret_cast<uint16_t*>(sm + L.kst);
  c.tmp = reinterpret_cast<uint32_t*>(sm + L.tmp);
  c.bval = reinterpret_cast<uint32_t*>(sm + L.bval);
  c.bidx = reinterpret_cast<int*>(sm + L.bidx);
  c.tval = reinterpret_cast<uint32_t*>(sm + L.tval);
  c.tidx = reinterpret_cast<int*>(sm + L.tidx);
  c.tval2 = reinterpret_cast<uint32_t*>(sm + L.tval2);
  c.tidx2 = reinterpret_cast<int*>(sm + L.tidx2);
  c.rank = reinterpret_cast<int*>(sm + L.rank);
  c.hist = reinterpret_cast<uint32_t*>(sm + L.hist);
  c.scal = reinterpret_cast<int*>(sm + L.scal);
  c.fscal = reinterpret_cast<float*>(sm + L.fscal);
  c.qstate = 0;
  c.kcap = s.Kb;
  return c;
}

// ---------------------------------------------------------------- a3 (shared by both kernels)
// F = the best min(cap, |M|) of the missing blocks M of S (ascending S of ns <= Kb
// entries, one per thread), written ascending to fetch[head].  se, cls, U, cblk
// hold at least Kb entries.
//
// diff_prepare lists M in S order in cblk[0..nM) with their scores in se[0..nM)
// and returns nM.  With se_all, se[x] already holds block x's score (the top-K
// pass loaded them); otherwise the scores are read from `scores`.
__device__ int diff_prepare(const Shape& s, const float2* scores, const int* S, int ns, const int* blk2slot,
                            int head, float2* se, int* cblk, int* red, bool se_all) {
  const int* b2s = blk2slot + (long long)head * s.nb_max;
  int x = -1, miss = 0;
  float2 sx = make_float2(0.f, 0.f);
  if ((int)threadIdx.x < ns) {
    x = S[threadIdx.x];
    miss = (x >= 0 && x < s.nb_max && b2s[x] < 0) ? 1 : 0;
    if (miss) sx = se_all ? se[x] : scores[(long long)head * s.nb_max + x];
  }
  // every se[x] is read before the scan's first barrier, every se[pos] written after
  const int pos = block_excl_scan(miss, red, red + 31);
  const int nM = red[31];
  if (miss) {
    cblk[pos] = x;
    se[pos] = sx;
  }
  __syncthreads();
  return nM;
}

// diff_emit writes the marked (cls == 1) entries of cblk[0..nM) to fetch[head] in
// order, pads with -1 and sets nfetch[head].  With host_kv (device address of
// the mapped host tier) each fetched block's 8 KiB is also prefetched into L2,
// so the gather that follows reads it there.
__device__ void diff_emit(const Shape& s, int nM, const uint8_t* cls, const int* cblk, int head, int* fetch,
                          int* nfetch, int* red, const uint16_t* host_kv) {
  int* out = fetch + (long long)head * s.Kb;
  const int take = ((int)threadIdx.x < nM && cls[threadIdx.x] == 1) ? 1 : 0;
  const int opos = block_excl_scan(take, red, red + 31);
  const int total = red[31];
  if (take && opos < s.Kb) out[opos] = cblk[threadIdx.x];
  if (take && host_kv) {
    const char* unit = reinterpret_cast<const char*>(host_kv + ((long long)head * s.nb_max + cblk[threadIdx.x]) *
                                                                   (2 * kBS * kD));
#pragma unroll 4
    for (int ln = 0; ln < 2 * kBS * kD * 2 / 128; ++ln)
      asm volatile("prefetch.global.L2 [%0];" ::"l"(unit + ln * 128));
  }
  for (int i = total + threadIdx.x; i < s.Kb; i += blockDim.x) out[i] = -1;
  if (threadIdx.x == 0) nfetch[head] = total < s.Kb ? total : s.Kb;
}

// ---------------------------------------------------------------- a2 kernel
// Pass 0 selects S (top-K of all nb blocks; every block when nb <= Kb) and writes
// it in ascending block order.  With kDiff, pass 1 runs a3 on that S in the same
// CTA (one launch for top-K and capped diff).  The passes form one loop that is
// not unrolled, so both run the same copy of the selection code and the second
// finds it in the instruction cache.
template <bool kPooled, bool kDiff, int NTH = kSelThreads>
__global__ void __launch_bounds__(NTH, 512 / NTH)
topk_select_kernel(Shape s, const float2* __restrict__ scores, const uint16_t* __restrict__ k_hbm,
                   const uint16_t* __restrict__ q_la, const int* __restrict__ ctx_len,
                   int* __restrict__ sel, int* __restrict__ nsel, const int* __restrict__ blk2slot, int cap,
                   int* __restrict__ fetch, int* __restrict__ nfetch, const uint16_t* __restrict__ host_kv,
                   TraceBuf tb) {
  TraceScope trace_(tb, OASIS_TRACE_SELECT);
  extern __shared__ __align__(16) char sm[];
  const SelLayout L = sel_layout(s.nb_max, kDiff, s.Kb, NTH / 32);
  const int head = blockIdx.x;
  const int b = head / s.Hkv;
  const int ctx = ctx_len[b];
  const int nb = clamp_nb(ctx, s.nb_max);
  int* out = sel + (long long)head * s.Kb;
  SelCtx c = make_ctx(sm, L, s, k_hbm, q_la, head, ctx, kPooled);
  float2* se = reinterpret_cast<float2*>(sm + L.se);
  uint8_t* cls = reinterpret_cast<uint8_t*>(sm + L.cls);
  int* U = reinterpret_cast<int*>(sm + L.U);
  int* red = reinterpret_cast<int*>(sm + L.red);
  int* cblk = reinterpret_cast<int*>(sm + L.cblk);
  const float2* src = scores + (long long)head * s.nb_max;
  {  // 16-byte loads (two entries) where the row allows, then the odd tail entry
    const int n2 = (((reinterpret_cast<uintptr_t>(src) & 15) == 0) ? nb : 0) >> 1;
    for (int i = threadIdx.x; i < n2; i += blockDim.x)
      reinterpret_cast<float4*>(se)[i] = reinterpret_cast<const float4*>(src)[i];
    for (int i = 2 * n2 + threadIdx.x; i < nb; i += blockDim.x) se[i] = src[i];
  }
  if (nb > s.Kb) issue_queries(c);
  if (kDiff) {  // the diff reads this head's blk2slot row after the top-K: bring it into L2 now
    const char* row = reinterpret_cast<const char*>(blk2slot + (long long)head * s.nb_max);
    for (int ln = threadIdx.x; ln * 128 < s.nb_max * 4; ln += blockDim.x)
      asm volatile("prefetch.global.L2 [%0];" ::"l"(row + ln * 128));
  }
  __syncthreads();
  int ns = 0;
#pragma unroll 1
  for (int pass = 0; pass < (kDiff ? 2 : 1); ++pass) {
    int n = nb, k = s.Kb;
    const int* cb = nullptr;
    if (pass == 1) {
      __syncthreads();  // the selection written by pass 0 is visible to the whole CTA
      n = diff_prepare(s, scores, out, ns, blk2slot, head, se, cblk, red, true);
      k = cap < n ? cap : n;
      cb = cblk;
    }
    select_best<kPooled>(c, se, n, k, cb, cls, U);
    if (pass == 0) {
      // compaction in ascending block order
      const int per = (nb + NTH - 1) / NTH;
      const int i0 = threadIdx.x * per, i1 = min(nb, i0 + per);
      int cnt = 0;
      for (int i = i0; i < i1; ++i) cnt += cls[i] == 1;
      int pos = block_excl_scan(cnt, red, red + 31);
      const int total = red[31];
      for (int i = i0; i < i1; ++i)
        if (cls[i] == 1) {
          if (pos < s.Kb) out[pos] = i;
          ++pos;
        }
      for (int i = total + threadIdx.x; i < s.Kb; i += blockDim.x) out[i] = -1;
      ns = total < s.Kb ? total : s.Kb;
      if (threadIdx.x == 0) nsel[head] = ns;
    } else {
      diff_emit(s, n, cls, cblk, head, fetch, nfetch, red, host_kv);
    }
  }
  if (c.qstate == 1) sel_cp_async_wait_all();  // no copy left in flight at exit
}

// ---------------------------------------------------------------- a3 kernel
template <bool kPooled>
__global__ void __launch_bounds__(kSelThreads, 2)
fetch_diff_kernel(Shape s, const float2* __restrict__ scores, const uint16_t* __restrict__ k_hbm,
                  const uint16_t* __restrict__ q_la, const int* __restrict__ ctx_len,
                  const int* __restrict__ sel, const int* __restrict__ nsel,
                  const int* __restrict__ blk2slot, int cap, int* __restrict__ fetch,
                  int* __restrict__ nfetch, TraceBuf tb) {
  TraceScope trace_(tb, OASIS_TRACE_SELECT);
  extern __shared__ __align__(16) char sm[];
  const SelLayout L = sel_layout(s.Kb, true, s.Kb);
  const int head = blockIdx.x;
  const int b = head / s.Hkv;
  const int ctx = ctx_len[b];
  SelCtx c = make_ctx(sm, L, s, k_hbm, q_la, head, ctx, kPooled);
  float2* se = reinterpret_cast<float2*>(sm + L.se);
  uint8_t* cls = reinterpret_cast<uint8_t*>(sm + L.cls);
  int* U = reinterpret_cast<int*>(sm + L.U);
  int* cblk = reinterpret_cast<int*>(sm + L.cblk);
  int* red = reinterpret_cast<int*>(sm + L.red);
  int ns = nsel[head];
  ns = ns < 0 ? 0 : (ns > s.Kb ? s.Kb : ns);
  issue_queries(c);
  const int nM = diff_prepare(s, scores, sel + (long long)head * s.Kb, ns, blk2slot, head, se, cblk, red, false);
  select_best<kPooled>(c, se, nM, cap < nM ? cap : nM, cblk, cls, U);
  diff_emit(s, nM, cls, cblk, head, fetch, nfetch, red, nullptr);
  if (c.qstate == 1) sel_cp_async_wait_all();  // no copy left in flight at exit
}

// ---------------------------------------------------------------- launchers
size_t topk_smem_bytes(const Shape& s) { return sel_layout(s.nb_max, false, s.Kb).total; }
size_t diff_smem_bytes(const Shape& s) { return sel_layout(s.Kb, true, s.Kb).total; }

template <bool kPooled, bool kDiff, int NTH>
static cudaError_t launch_topk_nth(const Shape& s, const float2* scores, const uint16_t* k, const uint16_t* q_la,
                                   const int* ctx, int* sel, int* nsel, cudaStream_t stream, const int* blk2slot,
                                   int cap, int* fetch, int* nfetch, const uint16_t* host_kv) {
  static int attr_cache[kMaxDevicesCached] = {};
  const size_t smem = sel_layout(s.nb_max, kDiff, s.Kb, NTH / 32).total;
  cudaError_t e = ensure_dyn_smem((const void*)topk_select_kernel<kPooled, kDiff, NTH>, smem, attr_cache);
  if (e != cudaSuccess) return e;
  topk_select_kernel<kPooled, kDiff, NTH><<<s.B * s.Hkv, NTH, smem, stream>>>(s, scores, k, q_la, ctx, sel, nsel,
                                                                              blk2slot, cap, fetch, nfetch, host_kv,
                                                                              trace_buf());
  return cudaGetLastError();
}

// Long candidate lists over few heads (at most one CTA per SM anyway) get 16 warps
// per head for the passes over all blocks; everything else 8 warps, two CTAs per SM.
template <bool kPooled, bool kDiff = false>
static cudaError_t launch_topk(const Shape& s, const float2* scores, const uint16_t* k, const uint16_t* q_la,
                               const int* ctx, int* sel, int* nsel, cudaStream_t stream,
                               const int* blk2slot = nullptr, int cap = 0, int* fetch = nullptr,
                               int* nfetch = nullptr, const uint16_t* host_kv = nullptr) {
  if constexpr (kDiff) {
    const bool wide = s.nb_max > 4096 && s.B * s.Hkv <= sm_count() &&
                      sel_layout(s.nb_max, kDiff, s.Kb, 16).total <= 227 * 1024;
    if (wide)
      return launch_topk_nth<kPooled, kDiff, 512>(s, scores, k, q_la, ctx, sel, nsel, stream, blk2slot, cap, fetch,
                                                  nfetch, host_kv);
  }
  return launch_topk_nth<kPooled, kDiff, kSelThreads>(s, scores, k, q_la, ctx, sel, nsel, stream, blk2slot, cap,
                                                      fetch, nfetch, host_kv);
}

cudaError_t launch_topk_select_diff(const Shape& s, const float2* scores, const uint16_t* k, const uint16_t* q_la,
                                    const int* ctx, const int* blk2slot, int cap, int* sel, int* nsel, int* fetch,
                                    int* nfetch, bool pooled, const uint16_t* host_kv, cudaStream_t stream) {
  return pooled ? launch_topk<true, true>(s, scores, k, q_la, ctx, sel, nsel, stream, blk2slot, cap, fetch, nfetch,
                                          host_kv)
                : launch_topk<false, true>(s, scores, k, q_la, ctx, sel, nsel, stream, blk2slot, cap, fetch, nfetch,
                                           host_kv);
}

template <bool kPooled>
static cudaError_t launch_diff(const Shape& s, const float2* scores, const uint16_t* k, const uint16_t* q_la,
                               const int* ctx, const int* sel, const int* nsel, const int* blk2slot, int cap,
                               int* fetch, int* nfetch, cudaStream_t stream) {
  static int attr_cache[kMaxDevicesCached] = {};
  const size_t smem = diff_smem_bytes(s);
  cudaError_t e = ensure_dyn_smem((const void*)fetch_diff_kernel<kPooled>, smem, attr_cache);
  if (e != cudaSuccess) return e;
  fetch_diff_kernel<kPooled><<<s.B * s.Hkv, kSelThreads, smem, stream>>>(s, scores, k, q_la, ctx, sel, nsel,
                                                                        blk2slot, cap, fetch, nfetch, trace_buf());
  return cudaGetLastError();
}

cudaError_t launch_topk_select(const Shape& s, const float2* scores, const uint16_t* k,
                               const uint16_t* q_la, const int* ctx, int* sel, int* nsel,
                               cudaStream_t stream) {
  return launch_topk<false>(s, scores, k, q_la, ctx, sel, nsel, stream);
}

cudaError_t launch_topk_select_pooled(const Shape& s, const float2* scores, const uint16_t* kp,
                                      const uint16_t* q_la, const int* ctx, int* sel, int* nsel,
                                      cudaStream_t stream) {
  return launch_topk<true>(s, scores, kp, q_la, ctx, sel, nsel, stream);
}

cudaError_t launch_fetch_diff(const Shape& s, const float2* scores, const uint16_t* k,
                              const uint16_t* q_la, const int* ctx, const int* sel,
                              const int* nsel, const int* blk2slot, int cap, int* fetch,
                              int* nfetch, cudaStream_t stream) {
  return launch_diff<false>(s, scores, k, q_la, ctx, sel, nsel, blk2slot, cap, fetch, nfetch, stream);
}

cudaError_t launch_fetch_diff_pooled(const Shape& s, const float2* scores, const uint16_t* kp,
                                     const uint16_t* q_la, const int* ctx, const int* sel,
                                     const int* nsel, const int* blk2slot, int cap, int* fetch,
                                     int* nfetch, cudaStream_t stream) {
  return launch_diff<true>(s, scores, kp, q_la, ctx, sel, nsel, blk2slot, cap, fetch, nfetch, stream);
}

}  // namespace oasis
