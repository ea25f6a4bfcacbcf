// f2: fused look-ahead attention - the true query and the lookahead (draft)
// queries of every head attend the same sparse KV in one pass.
//
// metalmedia.ai page, Figure 7 caption (right): the attention kernel processes
// the normal and the draft queries together over the sparse KV.  For KV head h
// of request b, A = { x in S : blk2slot[x] != -1 } as in a5, and each of its
// R = (1 + n_la) G query rows - row r < G is the true query of head hG + r, row
// G(1 + j) + g the lookahead query j of head hG + g - gets
//   softmax_t(scale * q_r . k_t) v_t over the valid tokens t of A (zero if none).
//
// Same structure as the a5 kernel (split-K over the entries of S, 4 warps each
// streaming every 4th resident block through a 2-stage cp.async ring) with all 16
// rows of the m16n8k16 tile in use: rows g and g+8 of a thread are two query
// rows, each with its own running max and sum.  Rows are grouped in m-tiles of
// 16 (grid z); a block's K and V are read once per m-tile, the second m-tile's
// reads normally hitting L2.
#include "common.cuh"

namespace oasis {

constexpr int kLaWarps = 4;
constexpr int kLaStage = 2 * kBS * kD * 2;                   // K + V of one block
constexpr int kLaSmem = kLaWarps * 2 * kLaStage;             // 64 KiB (reused for the warp merge)

__device__ __forceinline__ void la_cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void la_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void la_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }
__device__ __forceinline__ uint4 la_lds(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint32_t la_swz(int r, int c) { return (uint32_t)(r * 256 + ((c ^ (r & 7)) << 4)); }

// Query row rr (< R) of KV head h of request b.
__device__ __forceinline__ const uint16_t* la_qrow(const Shape& s, const uint16_t* q, const uint16_t* q_la, int b,
                                                   int h, int G, int rr) {
  if (rr < G) return q + ((long long)b * s.Hq + h * G + rr) * kD;
  const int j = rr / G - 1, gg = rr - (rr / G) * G;
  return q_la + (((long long)b * s.n_la + j) * s.Hq + h * G + gg) * kD;
}

__global__ void __launch_bounds__(kLaWarps * 32, 2)
attn_la_partial_kernel(Shape s, const uint16_t* __restrict__ q, const uint16_t* __restrict__ q_la,
                       const uint16_t* __restrict__ k_pool, const uint16_t* __restrict__ v_pool,
                       const int* __restrict__ sel, const int* __restrict__ nsel,
                       const int* __restrict__ blk2slot, const int* __restrict__ ctx_len, float scale_log2,
                       float* __restrict__ part_o, float* __restrict__ part_ml, int nsplit, int per_split) {
  extern __shared__ __align__(128) uint8_t lsm[];
  __shared__ float sm_m[kLaWarps][16];
  __shared__ float sm_l[kLaWarps][16];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int head = blockIdx.y, split = blockIdx.x, mt = blockIdx.z;
  const int b = head / s.Hkv, h = head - b * s.Hkv;
  const int G = s.Hq / s.Hkv;
  const int R = (1 + s.n_la) * G;
  int n = nsel[head];
  n = n < 0 ? 0 : (n > s.Kb ? s.Kb : n);
  const int ctx = ctx_len[b];
  const int p_begin = split * per_split;
  const int p_end = min(n, p_begin + per_split);
  const uint32_t ring = static_cast<uint32_t>(__cvta_generic_to_shared(lsm)) + warp * 2 * kLaStage;

  // A fragments of the two query rows of this thread (row g: qa0, row g + 8: qa1)
  const int r0 = mt * 16 + g, r1 = r0 + 8;
  uint32_t qa0[4][4], qa1[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint4 v0 = make_uint4(0u, 0u, 0u, 0u), v1 = v0;
    if (r0 < R) v0 = ldg_nc(la_qrow(s, q, q_la, b, h, G, r0) + (t + 4 * i) * 8);
    if (r1 < R) v1 = ldg_nc(la_qrow(s, q, q_la, b, h, G, r1) + (t + 4 * i) * 8);
    qa0[i][0] = v0.x; qa0[i][1] = v0.y; qa0[i][2] = v0.z; qa0[i][3] = v0.w;
    qa1[i][0] = v1.x; qa1[i][1] = v1.y; qa1[i][2] = v1.z; qa1[i][3] = v1.w;
  }

  float o[16][4];
#pragma unroll
  for (int j = 0; j < 16; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
  float m0 = neg_inf(), l0 = 0.f, m1 = neg_inf(), l1 = 0.f;
  const long long slot_base = (long long)head * s.P;

  for (int base = p_begin + warp; base < p_end; base += kLaWarps * 32) {
    const int p = base + kLaWarps * lane;
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
      const uint32_t dk = ring + st * kLaStage, dv = dk + kLaStage / 2;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int c = lane + 32 * j;
        const int r = c >> 4, cc = c & 15;
        la_cp_async16(dk + la_swz(r, cc), kb + r * kD + cc * 8);
        la_cp_async16(dv + la_swz(r, cc), vb + r * kD + cc * 8);
      }
      la_commit();
    };
    issue(0, cur);
    while (true) {
      const int nxt = mask ? __ffs(mask) - 1 : -1;
      if (nxt >= 0) {
        mask &= mask - 1;
        issue(stage ^ 1, nxt);
        la_wait<1>();
      } else {
        la_wait<0>();
      }
      __syncwarp();
      const int nt_cur = __shfl_sync(0xffffffffu, ntok, cur);
      const uint32_t dk = ring + stage * kLaStage, dv = dk + kLaStage / 2;
      // S = Q K^T: sc[nt][0,1] row g, sc[nt][2,3] row g+8; tokens nt*8 + 2t, +1
      float sc[2][4];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          const uint4 kv = la_lds(dk + la_swz(nt * 8 + g, t + 4 * i));
          const uint32_t kw[4] = {kv.x, kv.y, kv.z, kv.w};
#pragma unroll
          for (int hh = 0; hh < 2; ++hh)
            mma_bf16_16816(sc[nt][0], sc[nt][1], sc[nt][2], sc[nt][3], qa0[i][2 * hh], qa1[i][2 * hh],
                           qa0[i][2 * hh + 1], qa1[i][2 * hh + 1], kw[2 * hh], kw[2 * hh + 1]);
        }
      }
      float sv0[2][2], sv1[2][2];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const bool ok = nt * 8 + 2 * t + e < nt_cur;
          sv0[nt][e] = ok ? sc[nt][e] * scale_log2 : neg_inf();
          sv1[nt][e] = ok ? sc[nt][2 + e] * scale_log2 : neg_inf();
        }
      float bm0 = fmaxf(fmaxf(sv0[0][0], sv0[0][1]), fmaxf(sv0[1][0], sv0[1][1]));
      float bm1 = fmaxf(fmaxf(sv1[0][0], sv1[0][1]), fmaxf(sv1[1][0], sv1[1][1]));
      bm0 = fmaxf(bm0, __shfl_xor_sync(0xffffffffu, bm0, 1));
      bm0 = fmaxf(bm0, __shfl_xor_sync(0xffffffffu, bm0, 2));
      bm1 = fmaxf(bm1, __shfl_xor_sync(0xffffffffu, bm1, 1));
      bm1 = fmaxf(bm1, __shfl_xor_sync(0xffffffffu, bm1, 2));
      const float mn0 = fmaxf(m0, bm0), mn1 = fmaxf(m1, bm1);  // finite: token 0 is valid
      const float al0 = exp2f(m0 - mn0), al1 = exp2f(m1 - mn1);
      float pv0[2][2], pv1[2][2];
      float rs0 = 0.f, rs1 = 0.f;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          pv0[nt][e] = exp2f(sv0[nt][e] - mn0);
          pv1[nt][e] = exp2f(sv1[nt][e] - mn1);
          rs0 += pv0[nt][e];
          rs1 += pv1[nt][e];
        }
      rs0 += __shfl_xor_sync(0xffffffffu, rs0, 1);
      rs0 += __shfl_xor_sync(0xffffffffu, rs0, 2);
      rs1 += __shfl_xor_sync(0xffffffffu, rs1, 1);
      rs1 += __shfl_xor_sync(0xffffffffu, rs1, 2);
      l0 = l0 * al0 + rs0;
      l1 = l1 * al1 + rs1;
      m0 = mn0;
      m1 = mn1;
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        o[j][0] *= al0; o[j][1] *= al0;
        o[j][2] *= al1; o[j][3] *= al1;
      }
      // P as bf16 high part + bf16 residual; A operand rows g (a0, a2) and g+8 (a1, a3)
      const uint32_t h00 = pack_bf16x2(pv0[0][0], pv0[0][1]), h01 = pack_bf16x2(pv0[1][0], pv0[1][1]);
      const uint32_t h10 = pack_bf16x2(pv1[0][0], pv1[0][1]), h11 = pack_bf16x2(pv1[1][0], pv1[1][1]);
      const uint32_t e00 = pack_bf16x2(pv0[0][0] - bf_lo(h00), pv0[0][1] - bf_hi(h00));
      const uint32_t e01 = pack_bf16x2(pv0[1][0] - bf_lo(h01), pv0[1][1] - bf_hi(h01));
      const uint32_t e10 = pack_bf16x2(pv1[0][0] - bf_lo(h10), pv1[0][1] - bf_hi(h10));
      const uint32_t e11 = pack_bf16x2(pv1[1][0] - bf_lo(h11), pv1[1][1] - bf_hi(h11));
      uint4 vr[4][2];
      const int vrow[4] = {2 * t, 2 * t + 1, 2 * t + 8, 2 * t + 9};
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) vr[r][hf] = la_lds(dv + la_swz(vrow[r], 2 * g + hf));
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const uint32_t sel_half = (j & 1) ? 0x7632u : 0x5410u;
        const int wi = j >> 1;
        const uint32_t w0[4] = {vr[0][wi >> 2].x, vr[0][wi >> 2].y, vr[0][wi >> 2].z, vr[0][wi >> 2].w};
        const uint32_t w1[4] = {vr[1][wi >> 2].x, vr[1][wi >> 2].y, vr[1][wi >> 2].z, vr[1][wi >> 2].w};
        const uint32_t w2[4] = {vr[2][wi >> 2].x, vr[2][wi >> 2].y, vr[2][wi >> 2].z, vr[2][wi >> 2].w};
        const uint32_t w3[4] = {vr[3][wi >> 2].x, vr[3][wi >> 2].y, vr[3][wi >> 2].z, vr[3][wi >> 2].w};
        const uint32_t b0 = __byte_perm(w0[wi & 3], w1[wi & 3], sel_half);
        const uint32_t b1 = __byte_perm(w2[wi & 3], w3[wi & 3], sel_half);
        mma_bf16_16816(o[j][0], o[j][1], o[j][2], o[j][3], h00, h10, h01, h11, b0, b1);
        mma_bf16_16816(o[j][0], o[j][1], o[j][2], o[j][3], e00, e10, e01, e11, b0, b1);
      }
      __syncwarp();
      if (nxt < 0) break;
      cur = nxt;
      stage ^= 1;
    }
  }

  // merge the warps (ring reused: [kLaWarps][16 rows][kD] floats = 32 KiB)
  __syncthreads();
  float* sm_o = reinterpret_cast<float*>(lsm);
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    sm_o[(warp * 16 + g) * kD + 32 * t + j] = o[j][0];
    sm_o[(warp * 16 + g) * kD + 32 * t + 16 + j] = o[j][1];
    sm_o[(warp * 16 + g + 8) * kD + 32 * t + j] = o[j][2];
    sm_o[(warp * 16 + g + 8) * kD + 32 * t + 16 + j] = o[j][3];
  }
  if (t == 0) {
    sm_m[warp][g] = m0; sm_l[warp][g] = l0;
    sm_m[warp][g + 8] = m1; sm_l[warp][g + 8] = l1;
  }
  __syncthreads();
  const int MT = (R + 15) / 16;
  const long long pbase = (((long long)head * nsplit + split) * MT + mt) * 16;
  for (int idx = threadIdx.x; idx < 16 * kD; idx += blockDim.x) {
    const int rl = idx / kD, dd = idx - rl * kD;
    float M = neg_inf();
#pragma unroll
    for (int w = 0; w < kLaWarps; ++w) M = fmaxf(M, sm_m[w][rl]);
    float acc = 0.f, L = 0.f;
    if (M != neg_inf()) {
#pragma unroll
      for (int w = 0; w < kLaWarps; ++w) {
        const float f = exp2f(sm_m[w][rl] - M);
        acc += f * sm_o[(w * 16 + rl) * kD + dd];
        L += f * sm_l[w][rl];
      }
    }
    part_o[(pbase + rl) * kD + dd] = acc;
    if (dd == 0) {
      part_ml[(pbase + rl) * 2] = M;
      part_ml[(pbase + rl) * 2 + 1] = L;
    }
  }
}

// One warp per (head, query row < R): merge the splits, write out or out_la.
__global__ void __launch_bounds__(128)
attn_la_combine_kernel(Shape s, const float* __restrict__ part_o, const float* __restrict__ part_ml, int nsplit,
                       float* __restrict__ out, float* __restrict__ out_la) {
  const int lane = threadIdx.x & 31;
  const int G = s.Hq / s.Hkv;
  const int R = (1 + s.n_la) * G;
  const int MT = (R + 15) / 16;
  const long long row = (long long)blockIdx.x * 4 + (threadIdx.x >> 5);  // head * R + rr
  if (row >= (long long)s.B * s.Hkv * R) return;
  const long long head = row / R;
  const int rr = (int)(row - head * R);
  const int b = (int)(head / s.Hkv), h = (int)(head - (long long)b * s.Hkv);
  const int mt = rr >> 4, rl = rr & 15;
  float M = neg_inf();
  for (int sp = 0; sp < nsplit; ++sp) M = fmaxf(M, part_ml[(((head * nsplit + sp) * MT + mt) * 16 + rl) * 2]);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float L = 0.f;
  if (M != neg_inf()) {
    for (int sp = 0; sp < nsplit; ++sp) {
      const long long pr = ((head * nsplit + sp) * MT + mt) * 16 + rl;
      const float f = exp2f(part_ml[pr * 2] - M);
      L += f * part_ml[pr * 2 + 1];
      const float4 v = reinterpret_cast<const float4*>(part_o + pr * kD)[lane];
      acc.x += f * v.x; acc.y += f * v.y; acc.z += f * v.z; acc.w += f * v.w;
    }
  }
  const float inv = L > 0.f ? 1.0f / L : 0.f;
  float* dst;
  if (rr < G) {
    dst = out + ((long long)b * s.Hq + h * G + rr) * kD;
  } else {
    const int j = rr / G - 1, gg = rr - (rr / G) * G;
    dst = out_la + (((long long)b * s.n_la + j) * s.Hq + h * G + gg) * kD;
  }
  reinterpret_cast<float4*>(dst)[lane] = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
}

int attn_la_nsplit(const Shape& s) {
  const int G = s.Hq / s.Hkv;
  const int MT = ((1 + s.n_la) * G + 15) / 16;
  const int units = s.B * s.Hkv * MT;
  int ns = 2 * sm_count() / units;  // one resident wave, as for a5
  const int max_ns = (s.Kb + 3) / 4;
  if (ns > max_ns) ns = max_ns;
  return ns < 1 ? 1 : ns;
}

size_t attn_la_workspace_bytes(const Shape& s) {
  const int G = s.Hq / s.Hkv;
  const int MT = ((1 + s.n_la) * G + 15) / 16;
  const size_t rows = (size_t)s.B * s.Hkv * attn_la_nsplit(s) * MT * 16;
  return rows * kD * sizeof(float) + rows * 2 * sizeof(float);
}

cudaError_t launch_attn_lookahead(const Shape& s, const uint16_t* q, const uint16_t* q_la, const uint16_t* k_pool,
                                  const uint16_t* v_pool, const int* sel, const int* nsel, const int* blk2slot,
                                  const int* ctx, float scale, void* ws, float* out, float* out_la,
                                  cudaStream_t stream) {
  const int G = s.Hq / s.Hkv;
  const int R = (1 + s.n_la) * G;
  const int MT = (R + 15) / 16;
  const int nsplit = attn_la_nsplit(s);
  const int per_split = (s.Kb + nsplit - 1) / nsplit;
  const size_t rows = (size_t)s.B * s.Hkv * nsplit * MT * 16;
  float* part_o = static_cast<float*>(ws);
  float* part_ml = part_o + rows * kD;
  static int attr_cache[kMaxDevicesCached] = {};
  cudaError_t e = ensure_dyn_smem((const void*)attn_la_partial_kernel, kLaSmem, attr_cache);
  if (e != cudaSuccess) return e;
  const dim3 grid(nsplit, s.B * s.Hkv, MT);
  attn_la_partial_kernel<<<grid, kLaWarps * 32, kLaSmem, stream>>>(s, q, q_la, k_pool, v_pool, sel, nsel, blk2slot,
                                                                  ctx, scale * 1.4426950408889634f, part_o, part_ml,
                                                                  nsplit, per_split);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const long long nrows = (long long)s.B * s.Hkv * R;
  attn_la_combine_kernel<<<(unsigned)((nrows + 3) / 4), 128, 0, stream>>>(s, part_o, part_ml, nsplit, out, out_la);
  return cudaGetLastError();
}

}  // namespace oasis
