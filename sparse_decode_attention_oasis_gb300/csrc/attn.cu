// a5: block-sparse paged decode attention over the resident selected blocks.
//
// OasisKV abstract (attention over only the most relevant tokens kept in HBM) and
// metalmedia.ai page, Figure 7 caption, right (decode attention reads only the
// blocks selected and held on the GPU).  A = { x in S : blk2slot[x] != -1 }; for each query head
// of the GQA group, softmax(scale * q.k) v over the valid tokens of A.
//
// Split-K flash decode.  Grid (split, request*KV head); a split covers a range
// of entries of S and its 4 warps take every 4th entry.  A warp first looks up
// 32 entries at once (sel, then blk2slot: two rounds of loads), keeps the
// resident ones, and streams their K and V (8 KiB per block) through a 2-stage
// shared-memory ring with cp.async, so the next block is in flight while the
// current one is computed.  Rows are stored with their 16-byte chunks XOR-ed by
// (row mod 8) to spread the fragment reads over the banks.  Per block the warp
// computes S = Q K^T with the G query heads as the rows of one m16n8k16 tile
// (rows >= G are zero; the d axis is permuted identically for Q and K), runs the
// online softmax in fp32 (exp2 with scale*log2(e) folded in), and accumulates the
// output transposed, O^T += V^T P^T, so that the 16 rows of each MMA are 16 of
// the 128 output dimensions and the G queries its columns: the S accumulators
// of a thread are exactly its B fragment of P^T, and ldmatrix.trans reads V's
// A fragments straight from the staged rows.  Per block that is 8 d-slices x 2
// MMAs (P split into a bf16 high part and a bf16 residual, ~16 significant bits)
// and 32 fp32 accumulators per thread.  The 4 warps merge in shared memory; with
// one split the CTA writes the output, otherwise a second kernel merges the
// splits of each query head.
#include "common.cuh"

namespace oasis {

constexpr int kAttnWarps = 4;
constexpr int kStageBytes = 2 * kBS * kD * 2;                    // K + V of one block
constexpr int kAttnSmem = kAttnWarps * 2 * kStageBytes;          // 64 KiB

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// Four 8x8 b16 matrices, transposed: lane 8i + r gives the address of row r of
// matrix i; register i receives matrix i transposed (the A-fragment layout).
__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                              uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ uint4 lds_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}

// byte offset of 16-byte chunk c of row r in a staged 16 x 128 bf16 tile
__device__ __forceinline__ uint32_t swz(int r, int c) { return (uint32_t)(r * 256 + ((c ^ (r & 7)) << 4)); }

template <int G>
__global__ void __launch_bounds__(kAttnWarps * 32, 3)
attn_partial_kernel(Shape s, const uint16_t* __restrict__ q, const uint16_t* __restrict__ k_pool,
                    const uint16_t* __restrict__ v_pool, const int* __restrict__ sel,
                    const int* __restrict__ nsel, const int* __restrict__ blk2slot,
                    const int* __restrict__ ctx_len, float scale_log2, float* __restrict__ part_o,
                    float* __restrict__ part_ml, float* __restrict__ out, int nsplit, int per_split,
                    TraceBuf tb) {
  TraceScope trace_(tb, OASIS_TRACE_ATTN);
  extern __shared__ __align__(128) uint8_t asmem[];
  __shared__ float sm_m[kAttnWarps][G];
  __shared__ float sm_l[kAttnWarps][G];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int head = blockIdx.y, split = blockIdx.x;
  const int b = head / s.Hkv, h = head - b * s.Hkv;
  int n = nsel[head];
  n = n < 0 ? 0 : (n > s.Kb ? s.Kb : n);
  const int ctx = ctx_len[b];
  const int p_begin = split * per_split;
  const int p_end = min(n, p_begin + per_split);
  const uint32_t ring = static_cast<uint32_t>(__cvta_generic_to_shared(asmem)) + warp * 2 * kStageBytes;

  // Q fragments (rows g < G); chunk t+4i of the row gives words for k-steps 2i, 2i+1
  uint32_t qa[4][4];
  if (g < G) {
    const uint16_t* qrow = q + ((long long)b * s.Hq + h * G + g) * kD;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 v = ldg_nc(qrow + (t + 4 * i) * 8);
      qa[i][0] = v.x; qa[i][1] = v.y; qa[i][2] = v.z; qa[i][3] = v.w;
    }
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) qa[i][0] = qa[i][1] = qa[i][2] = qa[i][3] = 0u;
  }

  // O^T accumulators: slice m holds d = 16m + g (regs 0, 1) and 16m + g + 8
  // (regs 2, 3) for queries 2t and 2t + 1
  float o[8][4];
#pragma unroll
  for (int m = 0; m < 8; ++m) o[m][0] = o[m][1] = o[m][2] = o[m][3] = 0.f;
  // ldmatrix row of this lane: matrix i = lane / 8 covers tokens 8 (i / 2) .. + 7 and
  // the lower (i even) or upper 8 dimensions of a 16-wide slice
  const int lm_row = (lane & 7) + ((lane >> 4) << 3);
  const int lm_hi = (lane >> 3) & 1;
  float m_run = neg_inf(), l_run = 0.f;
  const long long slot_base = (long long)head * s.P;

  for (int base = p_begin + warp; base < p_end; base += kAttnWarps * 32) {
    // lane j looks up entry base + 4j
    const int p = base + kAttnWarps * lane;
    int slot = -1, ntok = 0;
    if (p < p_end) {
      const int x = sel[(long long)head * s.Kb + p];
      if (x >= 0 && x < s.nb_max) {
        const int sl = blk2slot[(long long)head * s.nb_max + x];
        ntok = min(kBS, ctx - x * kBS);
        if (sl >= 0 && sl < s.P && ntok > 0) slot = sl;
      }
    }
    unsigned mask = __ballot_sync(0xffffffffu, slot >= 0);
    if (!mask) continue;
    int stage = 0;
    int cur = __ffs(mask) - 1;
    mask &= mask - 1;
    auto issue = [&](int st, int src_lane) {
      const int sl = __shfl_sync(0xffffffffu, slot, src_lane);
      const uint16_t* kb = k_pool + (slot_base + sl) * kBS * kD;
      const uint16_t* vb = v_pool + (slot_base + sl) * kBS * kD;
      const uint32_t dk = ring + st * kStageBytes, dv = dk + kStageBytes / 2;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int c = lane + 32 * j;  // chunk of the 4 KiB tile
        const int r = c >> 4, cc = c & 15;
        cp_async16(dk + swz(r, cc), kb + r * kD + cc * 8);
        cp_async16(dv + swz(r, cc), vb + r * kD + cc * 8);
      }
      cp_async_commit();
    };
    issue(0, cur);
    while (true) {
      const int nxt = mask ? __ffs(mask) - 1 : -1;
      if (nxt >= 0) {
        mask &= mask - 1;
        issue(stage ^ 1, nxt);
        cp_async_wait<1>();
      } else {
        cp_async_wait<0>();
      }
      __syncwarp();
      const int nt_cur = __shfl_sync(0xffffffffu, ntok, cur);
      const uint32_t dk = ring + stage * kStageBytes, dv = dk + kStageBytes / 2;
      float sc[2][4];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          const uint4 kv = lds_v4(dk + swz(nt * 8 + g, t + 4 * i));
          const uint32_t kw[4] = {kv.x, kv.y, kv.z, kv.w};
#pragma unroll
          for (int hh = 0; hh < 2; ++hh)
            mma_bf16_16816(sc[nt][0], sc[nt][1], sc[nt][2], sc[nt][3], qa[i][2 * hh], 0u, qa[i][2 * hh + 1], 0u,
                           kw[2 * hh], kw[2 * hh + 1]);
        }
      }
      float sv[2][2];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int tok = nt * 8 + 2 * t + e;
          sv[nt][e] = tok < nt_cur ? sc[nt][e] * scale_log2 : neg_inf();
        }
      float bm = fmaxf(fmaxf(sv[0][0], sv[0][1]), fmaxf(sv[1][0], sv[1][1]));
      bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 1));
      bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 2));
      const float m_new = fmaxf(m_run, bm);  // finite: token 0 of the block is valid
      const float alpha = exp2f(m_run - m_new);
      float pv[2][2];
      float rs = 0.f;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          pv[nt][e] = exp2f(sv[nt][e] - m_new);
          rs += pv[nt][e];
        }
      rs += __shfl_xor_sync(0xffffffffu, rs, 1);
      rs += __shfl_xor_sync(0xffffffffu, rs, 2);
      l_run = l_run * alpha + rs;
      m_run = m_new;
      // alpha of this thread's output columns (queries 2t, 2t + 1), held by rows 2t, 2t + 1
      const float a0 = __shfl_sync(0xffffffffu, alpha, (2 * t) * 4);
      const float a1 = __shfl_sync(0xffffffffu, alpha, (2 * t + 1) * 4);
#pragma unroll
      for (int m = 0; m < 8; ++m) { o[m][0] *= a0; o[m][1] *= a1; o[m][2] *= a0; o[m][3] *= a1; }
      // B fragments of P^T (tokens x queries): tokens 2t, 2t+1 of n-tile 0 and 1 for query g
      const uint32_t ph0 = pack_bf16x2(pv[0][0], pv[0][1]);
      const uint32_t ph1 = pack_bf16x2(pv[1][0], pv[1][1]);
      const uint32_t pl0 = pack_bf16x2(pv[0][0] - bf_lo(ph0), pv[0][1] - bf_hi(ph0));
      const uint32_t pl1 = pack_bf16x2(pv[1][0] - bf_lo(ph1), pv[1][1] - bf_hi(ph1));
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        uint32_t v0, v1, v2, v3;  // A fragments of V^T for dimensions 16m .. 16m + 15
        ldsm_x4_trans(dv + swz(lm_row, 2 * m + lm_hi), v0, v1, v2, v3);
        mma_bf16_16816(o[m][0], o[m][1], o[m][2], o[m][3], v0, v1, v2, v3, ph0, ph1);
        mma_bf16_16816(o[m][0], o[m][1], o[m][2], o[m][3], v0, v1, v2, v3, pl0, pl1);
      }
      __syncwarp();  // the stage is refilled by the next issue
      if (nxt < 0) break;
      cur = nxt;
      stage ^= 1;
    }
  }

  // merge the warps of this split (the staging ring is reused for the partial outputs)
  __syncthreads();
  float* sm_o = reinterpret_cast<float*>(asmem);  // [kAttnWarps][G][kD]
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    const int qq = 2 * t + e;
    if (qq < G) {
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        sm_o[(warp * G + qq) * kD + 16 * m + g] = o[m][e];
        sm_o[(warp * G + qq) * kD + 16 * m + g + 8] = o[m][2 + e];
      }
    }
  }
  if (g < G && t == 0) { sm_m[warp][g] = m_run; sm_l[warp][g] = l_run; }
  __syncthreads();
  const long long pbase = ((long long)head * nsplit + split) * G;
  for (int idx = threadIdx.x; idx < G * kD; idx += blockDim.x) {
    const int gg = idx / kD, dd = idx - gg * kD;
    float M = neg_inf();
#pragma unroll
    for (int w = 0; w < kAttnWarps; ++w) M = fmaxf(M, sm_m[w][gg]);
    float acc = 0.f, L = 0.f;
    if (M != neg_inf()) {
#pragma unroll
      for (int w = 0; w < kAttnWarps; ++w) {
        const float f = exp2f(sm_m[w][gg] - M);
        acc += f * sm_o[(w * G + gg) * kD + dd];
        L += f * sm_l[w][gg];
      }
    }
    if (nsplit == 1) {
      out[((long long)b * s.Hq + h * G + gg) * kD + dd] = L > 0.f ? acc / L : 0.f;
    } else {
      part_o[(pbase + gg) * kD + dd] = acc;
      if (dd == 0) {
        part_ml[(pbase + gg) * 2] = M;
        part_ml[(pbase + gg) * 2 + 1] = L;
      }
    }
  }
}

// out[b][hq] = merge of the nsplit partial states of its KV head.
__global__ void __launch_bounds__(128)
attn_combine_kernel(Shape s, const float* __restrict__ part_o, const float* __restrict__ part_ml,
                    int nsplit, float* __restrict__ out) {
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * 4 + (threadIdx.x >> 5);  // b * Hq + hq
  if (row >= s.B * s.Hq) return;
  const int G = s.Hq / s.Hkv;
  const int b = row / s.Hq, hq = row - b * s.Hq;
  const int h = hq / G, gg = hq - h * G;
  const long long head = (long long)b * s.Hkv + h;
  float M = neg_inf();
  for (int sp = 0; sp < nsplit; ++sp) M = fmaxf(M, part_ml[((head * nsplit + sp) * G + gg) * 2]);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float L = 0.f;
  if (M != neg_inf()) {
    for (int sp = 0; sp < nsplit; ++sp) {
      const long long pr = (head * nsplit + sp) * G + gg;
      const float f = exp2f(part_ml[pr * 2] - M);
      L += f * part_ml[pr * 2 + 1];
      const float4 v = reinterpret_cast<const float4*>(part_o + pr * kD)[lane];
      acc.x += f * v.x; acc.y += f * v.y; acc.z += f * v.z; acc.w += f * v.w;
    }
  }
  const float inv = L > 0.f ? 1.0f / L : 0.f;
  reinterpret_cast<float4*>(out + (long long)row * kD)[lane] =
      make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
}

// Splits per head: as many as keep the whole grid resident at once (2 CTAs per
// SM counted, though three fit), each split holding at least 4 entries of S.
// A second wave would double the latency chain; a warp with more blocks keeps
// its 2-stage ring busy instead.
int attn_nsplit(const Shape& s) {
  const int heads = s.B * s.Hkv;
  const int resident = 2 * sm_count();
  int ns = resident / heads;
  const int max_ns = (s.Kb + 3) / 4;
  if (ns > max_ns) ns = max_ns;
  return ns < 1 ? 1 : ns;
}

size_t attn_workspace_bytes(const Shape& s) {
  const size_t rows = (size_t)s.B * s.Hkv * attn_nsplit(s) * (s.Hq / s.Hkv);
  return rows * kD * sizeof(float) + rows * 2 * sizeof(float);
}

cudaError_t launch_sparse_decode_attn(const Shape& s, const uint16_t* q, const uint16_t* k_pool,
                                      const uint16_t* v_pool, const int* sel, const int* nsel,
                                      const int* blk2slot, const int* ctx, float scale, void* ws,
                                      float* out, cudaStream_t stream) {
  const int nsplit = attn_nsplit(s);
  const int per_split = (s.Kb + nsplit - 1) / nsplit;
  const int G = s.Hq / s.Hkv;
  const size_t rows = (size_t)s.B * s.Hkv * nsplit * G;
  float* part_o = static_cast<float*>(ws);
  float* part_ml = part_o + rows * kD;
  const float scale_log2 = scale * 1.4426950408889634f;
  dim3 grid(nsplit, s.B * s.Hkv);
  dim3 block(kAttnWarps * 32);
  static int attr_cache[4][kMaxDevicesCached] = {};
  cudaError_t e = cudaSuccess;
  const TraceBuf tb = trace_buf();
#define OASIS_ATTN_LAUNCH(GG, IDX)                                                                              \
  e = ensure_dyn_smem((const void*)attn_partial_kernel<GG>, kAttnSmem, attr_cache[IDX]);                      \
  if (e != cudaSuccess) return e;                                                                              \
  attn_partial_kernel<GG><<<grid, block, kAttnSmem, stream>>>(s, q, k_pool, v_pool, sel, nsel, blk2slot, ctx,  \
                                                              scale_log2, part_o, part_ml, out, nsplit,       \
                                                              per_split, tb);
  switch (G) {
    case 1: OASIS_ATTN_LAUNCH(1, 0) break;
    case 2: OASIS_ATTN_LAUNCH(2, 1) break;
    case 4: OASIS_ATTN_LAUNCH(4, 2) break;
    case 8: OASIS_ATTN_LAUNCH(8, 3) break;
    default: return cudaErrorInvalidValue;
  }
#undef OASIS_ATTN_LAUNCH
  e = cudaGetLastError();
  if (e != cudaSuccess || nsplit == 1) return e;
  const int rowsq = s.B * s.Hq;
  attn_combine_kernel<<<(rowsq + 3) / 4, 128, 0, stream>>>(s, part_o, part_ml, nsplit, out);
  return cudaGetLastError();
}

}  // namespace oasis
