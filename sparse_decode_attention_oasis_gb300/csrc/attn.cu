// a5: block-sparse paged decode attention over the resident selected blocks.
//
// OasisKV abstract (attention over only the most relevant tokens kept in HBM) and
// metalmedia.ai page, Figure 7 caption, right (decode attention reads only the
// blocks selected and held on the GPU).  A = { x in S : blk2slot[x] != -1 }; for each query head
// of the GQA group, softmax(scale * q.k) v over the valid tokens of A.
//
// Split-K flash decode.  Grid (split, request*KV head); a split covers
// kAttnSplit consecutive entries of S, 4 warps take kAttnPerWarp each.  Per
// 16-token block a warp computes S = Q K^T with the G query heads as the rows of
// one m16n8k16 tile (rows >= G are zero), runs the online softmax in fp32 (exp2
// with scale*log2(e) folded in), and accumulates O += P V where P is split into
// a bf16 high part and a bf16 residual (two MMAs), so the weights carry ~16
// significant bits.  K rows are loaded as B fragments straight from HBM with the
// same d permutation as the Q fragments; V rows are loaded as 32-byte row
// segments and re-paired into B fragments with byte permutes, the output column
// of n-tile j / column n being d = 16 n + j.  The 4 warps merge in shared memory;
// a second kernel merges the splits of each query head.
#include "common.cuh"

namespace oasis {

constexpr int kAttnWarps = 4;
constexpr int kAttnPerWarp = 4;
constexpr int kAttnSplit = kAttnWarps * kAttnPerWarp;  // 16 blocks = 256 tokens per CTA

template <int G>
__global__ void __launch_bounds__(kAttnWarps * 32, 3)
attn_partial_kernel(Shape s, const uint16_t* __restrict__ q, const uint16_t* __restrict__ k_pool,
                    const uint16_t* __restrict__ v_pool, const int* __restrict__ sel,
                    const int* __restrict__ nsel, const int* __restrict__ blk2slot,
                    const int* __restrict__ ctx_len, float scale_log2, float* __restrict__ part_o,
                    float* __restrict__ part_ml, int nsplit) {
  __shared__ float sm_o[kAttnWarps][G][kD];
  __shared__ float sm_m[kAttnWarps][G];
  __shared__ float sm_l[kAttnWarps][G];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int head = blockIdx.y, split = blockIdx.x;
  const int b = head / s.Hkv, h = head - b * s.Hkv;
  int n = nsel[head];
  n = n < 0 ? 0 : (n > s.Kb ? s.Kb : n);
  const int ctx = ctx_len[b];
  const int p0 = split * kAttnSplit + warp * kAttnPerWarp;
  const int p1 = min(n, p0 + kAttnPerWarp);

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

  float o[16][4];
#pragma unroll
  for (int j = 0; j < 16; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
  float m_run = neg_inf(), l_run = 0.f;

  const long long slot_base = (long long)head * s.P;
  for (int p = p0; p < p1; ++p) {
    const int x = sel[(long long)head * s.Kb + p];
    if (x < 0 || x >= s.nb_max) continue;
    const int slot = blk2slot[(long long)head * s.nb_max + x];
    if (slot < 0 || slot >= s.P) continue;
    const int ntok = min(kBS, ctx - x * kBS);
    if (ntok <= 0) continue;
    const uint16_t* kb = k_pool + (slot_base + slot) * kBS * kD;
    const uint16_t* vb = v_pool + (slot_base + slot) * kBS * kD;
    uint4 kr[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int i = 0; i < 4; ++i) kr[nt][i] = ldg_stream(kb + (nt * 8 + g) * kD + (t + 4 * i) * 8);
    uint4 vr[4][2];
    const int vrow[4] = {2 * t, 2 * t + 1, 2 * t + 8, 2 * t + 9};
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) vr[r][hf] = ldg_stream(vb + vrow[r] * kD + 16 * g + 8 * hf);

    float sc[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          const uint32_t kw[4] = {kr[nt][i].x, kr[nt][i].y, kr[nt][i].z, kr[nt][i].w};
          mma_bf16_16816(sc[nt][0], sc[nt][1], sc[nt][2], sc[nt][3], qa[i][2 * hh], 0u,
                         qa[i][2 * hh + 1], 0u, kw[2 * hh], kw[2 * hh + 1]);
        }
      }
    }
    // row g: tokens nt*8 + 2t + {0,1}
    float sv[2][2];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int tok = nt * 8 + 2 * t + e;
        sv[nt][e] = tok < ntok ? sc[nt][e] * scale_log2 : neg_inf();
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
#pragma unroll
    for (int j = 0; j < 16; ++j) { o[j][0] *= alpha; o[j][1] *= alpha; }
    const uint32_t ph0 = pack_bf16x2(pv[0][0], pv[0][1]);
    const uint32_t ph1 = pack_bf16x2(pv[1][0], pv[1][1]);
    const uint32_t pl0 = pack_bf16x2(pv[0][0] - bf_lo(ph0), pv[0][1] - bf_hi(ph0));
    const uint32_t pl1 = pack_bf16x2(pv[1][0] - bf_lo(ph1), pv[1][1] - bf_hi(ph1));
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
      mma_bf16_16816(o[j][0], o[j][1], o[j][2], o[j][3], ph0, 0u, ph1, 0u, b0, b1);
      mma_bf16_16816(o[j][0], o[j][1], o[j][2], o[j][3], pl0, 0u, pl1, 0u, b0, b1);
    }
  }

  // merge the warps of this split
  if (g < G) {
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      sm_o[warp][g][32 * t + j] = o[j][0];
      sm_o[warp][g][32 * t + 16 + j] = o[j][1];
    }
    if (t == 0) { sm_m[warp][g] = m_run; sm_l[warp][g] = l_run; }
  }
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
        acc += f * sm_o[w][gg][dd];
        L += f * sm_l[w][gg];
      }
    }
    part_o[(pbase + gg) * kD + dd] = acc;
    if (dd == 0) {
      part_ml[(pbase + gg) * 2] = M;
      part_ml[(pbase + gg) * 2 + 1] = L;
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

int attn_nsplit(const Shape& s) { return (s.Kb + kAttnSplit - 1) / kAttnSplit; }

size_t attn_workspace_bytes(const Shape& s) {
  const size_t rows = (size_t)s.B * s.Hkv * attn_nsplit(s) * (s.Hq / s.Hkv);
  return rows * kD * sizeof(float) + rows * 2 * sizeof(float);
}

cudaError_t launch_sparse_decode_attn(const Shape& s, const uint16_t* q, const uint16_t* k_pool,
                                      const uint16_t* v_pool, const int* sel, const int* nsel,
                                      const int* blk2slot, const int* ctx, float scale, void* ws,
                                      float* out, cudaStream_t stream) {
  const int nsplit = attn_nsplit(s);
  const int G = s.Hq / s.Hkv;
  const size_t rows = (size_t)s.B * s.Hkv * nsplit * G;
  float* part_o = static_cast<float*>(ws);
  float* part_ml = part_o + rows * kD;
  const float scale_log2 = scale * 1.4426950408889634f;
  dim3 grid(nsplit, s.B * s.Hkv);
  dim3 block(kAttnWarps * 32);
  switch (G) {
    case 1: attn_partial_kernel<1><<<grid, block, 0, stream>>>(s, q, k_pool, v_pool, sel, nsel, blk2slot, ctx, scale_log2, part_o, part_ml, nsplit); break;
    case 2: attn_partial_kernel<2><<<grid, block, 0, stream>>>(s, q, k_pool, v_pool, sel, nsel, blk2slot, ctx, scale_log2, part_o, part_ml, nsplit); break;
    case 4: attn_partial_kernel<4><<<grid, block, 0, stream>>>(s, q, k_pool, v_pool, sel, nsel, blk2slot, ctx, scale_log2, part_o, part_ml, nsplit); break;
    case 8: attn_partial_kernel<8><<<grid, block, 0, stream>>>(s, q, k_pool, v_pool, sel, nsel, blk2slot, ctx, scale_log2, part_o, part_ml, nsplit); break;
    default: return cudaErrorInvalidValue;
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int rowsq = s.B * s.Hq;
  attn_combine_kernel<<<(rowsq + 3) / 4, 128, 0, stream>>>(s, part_o, part_ml, nsplit, out);
  return cudaGetLastError();
}

}  // namespace oasis
