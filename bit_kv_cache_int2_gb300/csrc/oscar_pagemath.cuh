// INT2 page math on mma.sync tensor-core fragments, shared by the decode
// kernels (sm_103a).  The decode paragraph under the pipeline figure
// "从离线校准到在线推理的pipeline" of "超越TurboQuant：Together AI把2-bit KV Cache推向
// 真实服务": the INT2 history is unpacked, dequantised with its scale / zero
// point and accumulated in floating point, with online softmax across pages.
#pragma once

#include "oscar_internal.cuh"

namespace oscar {

constexpr int DEC_NW = 4;  // warps per decode CTA

// max(a, b, c) in one instruction.
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// ------------------------------------------------- per-warp decode state
template <int NG>
struct Int2State {
  float oacc[8][4];  // o'^T: m-tile j, rows channels 16j+gid / 16j+8+gid, cols heads 2tq, 2tq+1
  float m[2];        // running max (log2 units) of heads 2tq, 2tq+1
  float l[2];        // this thread's part of the running sum
  float zs[2][NG];   // this thread's part of sum p * z_v
  uint32_t bq[8][2];  // q' B fragments (column = head gid)
  float ka[2];        // logit scale per column head
  float kb[2][NG];    // logit offset per column head and group (codebook pages only)
  float kg[2][NG];    // z-term weight per column head and group
};

// One INT2 page (64 tokens) of one kv head on tensor cores.  stage: the page's
// head block in smem; nv: valid tokens.
template <int NG, bool FULL>
__device__ __forceinline__ void int2_page_mma(Int2State<NG>& S, const uint8_t* stage, int nv,
                                              int lane) {
  const int gid = lane >> 2, tq = lane & 3;
  constexpr int KPG = 8 / NG;   // k-steps per group (QK)
  constexpr int MPG = 8 / NG;   // m-tiles per group (SV)
  const uint8_t* kc = stage;
  const uint8_t* vc = stage + 2048;
  const __half2* ksz = (const __half2*)(stage + 4096);
  const __half2* vsz = (const __half2*)(stage + 4096 + PAGE * NG * 4);

  // QK^T of the 4 tiles with the tiles interleaved, so that the 4
  // accumulator chains are independent
  uint2 wa[4], wb[4];
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    wa[s] = *(const uint2*)(kc + (16 * s + gid) * 32 + 8 * tq);
    wb[s] = *(const uint2*)(kc + (16 * s + gid + 8) * 32 + 8 * tq);
  }
  float acc[4][NG][4];
#pragma unroll
  for (int s = 0; s < 4; ++s)
#pragma unroll
    for (int gr = 0; gr < NG; ++gr) acc[s][gr][0] = acc[s][gr][1] = acc[s][gr][2] = acc[s][gr][3] = 0.f;
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      const uint32_t xa = kk < 4 ? wa[s].x : wa[s].y;
      const uint32_t xb = kk < 4 ? wb[s].x : wb[s].y;
      uint32_t a0, a1, a2, a3;
      switch (kk & 3) {
        case 0: a0 = code_sub<0>(xa); a1 = code_sub<0>(xb); a2 = code_sub<1>(xa); a3 = code_sub<1>(xb); break;
        case 1: a0 = code_sub<2>(xa); a1 = code_sub<2>(xb); a2 = code_sub<3>(xa); a3 = code_sub<3>(xb); break;
        case 2: a0 = code_sub<4>(xa); a1 = code_sub<4>(xb); a2 = code_sub<5>(xa); a3 = code_sub<5>(xb); break;
        default: a0 = code_sub<6>(xa); a1 = code_sub<6>(xb); a2 = code_sub<7>(xa); a3 = code_sub<7>(xb); break;
      }
      mma_f16(acc[s][kk / KPG], a0, a1, a2, a3, S.bq[kk][0], S.bq[kk][1]);
    }
  }
  float lam[4][4];
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    const int ta = 16 * s + gid, tb = ta + 8;
    // logits (log2 units): sum_gr s*(acc*alpha + beta) + z*gamma
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int row = e < 2 ? ta : tb;
      const int hc = e & 1;
      float v = 0.f;
#pragma unroll
      for (int gr = 0; gr < NG; ++gr) {
        const float2 sz = __half22float2(ksz[row * NG + gr]);
        v = fmaf(sz.x, acc[s][gr][e] * S.ka[hc], fmaf(sz.y, S.kg[hc][gr], v));
      }
      lam[s][e] = (FULL || row < nv) ? v : -INFINITY;
    }
  }
  // page max per column head, over all 64 tokens
  float pm[2] = {-INFINITY, -INFINITY};
#pragma unroll
  for (int s = 0; s < 4; ++s)
#pragma unroll
    for (int e = 0; e < 4; ++e) pm[e & 1] = fmaxf(pm[e & 1], lam[s][e]);
#pragma unroll
  for (int hc = 0; hc < 2; ++hc) {
    pm[hc] = fmaxf(pm[hc], __shfl_xor_sync(0xffffffffu, pm[hc], 4));
    pm[hc] = fmaxf(pm[hc], __shfl_xor_sync(0xffffffffu, pm[hc], 8));
    pm[hc] = fmaxf(pm[hc], __shfl_xor_sync(0xffffffffu, pm[hc], 16));
  }
  // rescale the running sums only when some lane's maximum moved
  {
    const float mn0 = fmaxf(S.m[0], pm[0]), mn1 = fmaxf(S.m[1], pm[1]);
    const bool moved = (mn0 > S.m[0]) || (mn1 > S.m[1]);
    if (__any_sync(0xffffffffu, moved)) {
      const float al0 = ex2(S.m[0] - mn0), al1 = ex2(S.m[1] - mn1);
      S.m[0] = mn0;
      S.m[1] = mn1;
      S.l[0] *= al0;
      S.l[1] *= al1;
#pragma unroll
      for (int gr = 0; gr < NG; ++gr) {
        S.zs[0][gr] *= al0;
        S.zs[1][gr] *= al1;
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        S.oacc[j][0] *= al0;
        S.oacc[j][2] *= al0;
        S.oacc[j][1] *= al1;
        S.oacc[j][3] *= al1;
      }
    }
  }
  // V code words: rows 16j+gid and 16j+8+gid, word tq (all 4 tiles)
  uint32_t vw[8][2];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    vw[j][0] = *(const uint32_t*)(vc + (16 * j + gid) * 16 + 4 * tq);
    vw[j][1] = *(const uint32_t*)(vc + (16 * j + 8 + gid) * 16 + 4 * tq);
  }
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    const int ta = 16 * s + gid, tb = ta + 8;
    const bool va = FULL || ta < nv, vb = FULL || tb < nv;
    float p[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      p[e] = ex2(lam[s][e] - S.m[e & 1]);
      S.l[e & 1] += p[e];
    }
    // scale of the code's bit position: rows < 8 use bit pair 2s, rows >= 8 use 2s+1
    const float fa = (float)(1 << (8 - code_exp_rt(2 * s)));
    const float fb = (float)(1 << (8 - code_exp_rt(2 * s + 1)));
#pragma unroll
    for (int gr = 0; gr < NG; ++gr) {
      const float2 sa = __half22float2(vsz[ta * NG + gr]);
      const float2 sb = __half22float2(vsz[tb * NG + gr]);
      const float s_a = va ? sa.x * fa : 0.f, z_a = va ? sa.y : 0.f;
      const float s_b = vb ? sb.x * fb : 0.f, z_b = vb ? sb.y : 0.f;
      const __half2 h0 = __floats2half2_rn(p[0] * s_a, p[1] * s_a);
      const __half2 h1 = __floats2half2_rn(p[2] * s_b, p[3] * s_b);
      S.zs[0][gr] = fmaf(p[0], z_a, fmaf(p[2], z_b, S.zs[0][gr]));
      S.zs[1][gr] = fmaf(p[1], z_a, fmaf(p[3], z_b, S.zs[1][gr]));
      const uint32_t b0 = movmatrix_t(*(const uint32_t*)&h0);
      const uint32_t b1 = movmatrix_t(*(const uint32_t*)&h1);
#pragma unroll
      for (int jj = 0; jj < MPG; ++jj) {
        const int j = gr * MPG + jj;
        uint32_t a0, a1, a2, a3;
        switch (s) {
          case 0: a0 = code_sub<0>(vw[j][0]); a1 = code_sub<0>(vw[j][1]); a2 = code_sub<1>(vw[j][0]); a3 = code_sub<1>(vw[j][1]); break;
          case 1: a0 = code_sub<2>(vw[j][0]); a1 = code_sub<2>(vw[j][1]); a2 = code_sub<3>(vw[j][0]); a3 = code_sub<3>(vw[j][1]); break;
          case 2: a0 = code_sub<4>(vw[j][0]); a1 = code_sub<4>(vw[j][1]); a2 = code_sub<5>(vw[j][0]); a3 = code_sub<5>(vw[j][1]); break;
          default: a0 = code_sub<6>(vw[j][0]); a1 = code_sub<6>(vw[j][1]); a2 = code_sub<7>(vw[j][0]); a3 = code_sub<7>(vw[j][1]); break;
        }
        mma_f16(S.oacc[j], a0, a1, a2, a3, b0, b1);
      }
    }
  }
}

// ------------------------------------- two INT2 pages as two streams (G <= 4)
// With at most 4 query heads per kv head, half of the m16n8 tile's columns
// would carry padding.  Instead a warp takes its pages two at a time: page A's
// logits fill columns 0..3 and page B's columns 4..7 of the same QK^T tile,
// each column keeps its own online-softmax state, and the SV^T products read
// the shared P tile with the other page's columns masked to zero.  Column n
// of the B operands lives in the lanes with gid == n, so the masks are
// per-lane constants: mA = all ones where gid < 4.  At the end of an item the
// two streams of a head (columns n and n + 4, lanes tq and tq ^ 2) are merged.
// The codes enter as fp16 subnormals (code_sub): the products carry no
// offset, so the running sums of B that the offset form needs are not kept.
// The caller's constants: logit scale ka = 2^24 * alpha of the packed query
// record and no logit offset; the output is 2^16 * O + (sum of p z).
template <int NG>
__device__ __forceinline__ void qk_page_masked(float (&acc)[4][NG][4], const uint8_t* kc,
                                               const uint32_t (&bq)[8][2], uint32_t mask, int gid,
                                               int tq) {
  constexpr int KPG = 8 / NG;
  uint2 wa[4], wb[4];
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    wa[s] = *(const uint2*)(kc + (16 * s + gid) * 32 + 8 * tq);
    wb[s] = *(const uint2*)(kc + (16 * s + gid + 8) * 32 + 8 * tq);
  }
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    const uint32_t b0 = bq[kk][0] & mask, b1 = bq[kk][1] & mask;
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      const uint32_t xa = kk < 4 ? wa[s].x : wa[s].y;
      const uint32_t xb = kk < 4 ? wb[s].x : wb[s].y;
      uint32_t a0, a1, a2, a3;
      switch (kk & 3) {
        case 0: a0 = code_sub<0>(xa); a1 = code_sub<0>(xb); a2 = code_sub<1>(xa); a3 = code_sub<1>(xb); break;
        case 1: a0 = code_sub<2>(xa); a1 = code_sub<2>(xb); a2 = code_sub<3>(xa); a3 = code_sub<3>(xb); break;
        case 2: a0 = code_sub<4>(xa); a1 = code_sub<4>(xb); a2 = code_sub<5>(xa); a3 = code_sub<5>(xb); break;
        default: a0 = code_sub<6>(xa); a1 = code_sub<6>(xb); a2 = code_sub<7>(xa); a3 = code_sub<7>(xb); break;
      }
      mma_f16(acc[s][kk / KPG], a0, a1, a2, a3, b0, b1);
    }
  }
}

template <int NG, bool FULL>
__device__ __forceinline__ void int2_pair_mma(Int2State<NG>& S, const uint8_t* stA, int nvA,
                                              const uint8_t* stB, int nvB, bool hasB, int lane,
                                              uint32_t mA) {
  const int gid = lane >> 2, tq = lane & 3;
  constexpr int MPG = 8 / NG;
  float acc[4][NG][4];
#pragma unroll
  for (int s = 0; s < 4; ++s)
#pragma unroll
    for (int gr = 0; gr < NG; ++gr) acc[s][gr][0] = acc[s][gr][1] = acc[s][gr][2] = acc[s][gr][3] = 0.f;
  const uint32_t mB = ~mA;
  qk_page_masked<NG>(acc, stA, S.bq, mA, gid, tq);
  // page B's products run even when there is no page B, with its B operand
  // masked to zero: no branch around the tensor-core instructions
  const uint32_t mBB = hasB ? mB : 0u;
  qk_page_masked<NG>(acc, stB, S.bq, mBB, gid, tq);
  // this lane's columns 2tq, 2tq + 1 belong to page A when tq < 2
  const bool own_a = tq < 2;
  const uint8_t* st = own_a ? stA : stB;
  const int nv = own_a ? nvA : nvB;
  const __half2* ksz = (const __half2*)(st + 4096);
  const __half2* vsz = (const __half2*)(st + 4096 + PAGE * NG * 4);
  float lam[4][4];
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    const int ta = 16 * s + gid, tb = ta + 8;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int row = e < 2 ? ta : tb;
      const int hc = e & 1;
      float v = 0.f;
#pragma unroll
      for (int gr = 0; gr < NG; ++gr) {
        const float2 sz = __half22float2(ksz[row * NG + gr]);
        v = fmaf(sz.x, acc[s][gr][e] * S.ka[hc], fmaf(sz.y, S.kg[hc][gr], v));
      }
      lam[s][e] = v;
    }
  }
  if (!FULL && (nvA < PAGE || nvB < PAGE)) {  // warp-uniform: a partial page or no page B
#pragma unroll
    for (int s = 0; s < 4; ++s)
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if ((e < 2 ? 16 * s + gid : 16 * s + gid + 8) >= nv) lam[s][e] = -INFINITY;
  }
  float pm[2];
#pragma unroll
  for (int hc = 0; hc < 2; ++hc) {
    float x = fmax3(lam[0][hc], lam[0][hc + 2], lam[1][hc]);
    float y = fmax3(lam[1][hc + 2], lam[2][hc], lam[2][hc + 2]);
    pm[hc] = fmax3(x, y, fmaxf(lam[3][hc], lam[3][hc + 2]));
  }
#pragma unroll
  for (int hc = 0; hc < 2; ++hc) {
    pm[hc] = fmaxf(pm[hc], __shfl_xor_sync(0xffffffffu, pm[hc], 4));
    pm[hc] = fmaxf(pm[hc], __shfl_xor_sync(0xffffffffu, pm[hc], 8));
    pm[hc] = fmaxf(pm[hc], __shfl_xor_sync(0xffffffffu, pm[hc], 16));
  }
  {
    const float mn0 = fmaxf(S.m[0], pm[0]), mn1 = fmaxf(S.m[1], pm[1]);
    const bool moved = (mn0 > S.m[0]) || (mn1 > S.m[1]);
    if (__any_sync(0xffffffffu, moved)) {
      const float al0 = ex2(S.m[0] - mn0), al1 = ex2(S.m[1] - mn1);
      S.m[0] = mn0;
      S.m[1] = mn1;
      S.l[0] *= al0;
      S.l[1] *= al1;
#pragma unroll
      for (int gr = 0; gr < NG; ++gr) {
        S.zs[0][gr] *= al0;
        S.zs[1][gr] *= al1;
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        S.oacc[j][0] *= al0;
        S.oacc[j][2] *= al0;
        S.oacc[j][1] *= al1;
        S.oacc[j][3] *= al1;
      }
    }
  }
  const uint8_t* vcA = stA + 2048;
  const uint8_t* vcB = stB + 2048;
  uint32_t va_w[8][2], vb_w[8][2];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    va_w[j][0] = *(const uint32_t*)(vcA + (16 * j + gid) * 16 + 4 * tq);
    va_w[j][1] = *(const uint32_t*)(vcA + (16 * j + 8 + gid) * 16 + 4 * tq);
    vb_w[j][0] = *(const uint32_t*)(vcB + (16 * j + gid) * 16 + 4 * tq);
    vb_w[j][1] = *(const uint32_t*)(vcB + (16 * j + 8 + gid) * 16 + 4 * tq);
  }
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    const int ta = 16 * s + gid, tb = ta + 8;
    const bool va = FULL || ta < nv, vb = FULL || tb < nv;
    float p[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      p[e] = ex2(lam[s][e] - S.m[e & 1]);
      S.l[e & 1] += p[e];
    }
    const float fa = (float)(1 << (8 - code_exp_rt(2 * s)));
    const float fb = (float)(1 << (8 - code_exp_rt(2 * s + 1)));
#pragma unroll
    for (int gr = 0; gr < NG; ++gr) {
      const float2 sa = __half22float2(vsz[ta * NG + gr]);
      const float2 sb = __half22float2(vsz[tb * NG + gr]);
      const float s_a = va ? sa.x * fa : 0.f, z_a = va ? sa.y : 0.f;
      const float s_b = vb ? sb.x * fb : 0.f, z_b = vb ? sb.y : 0.f;
      const __half2 h0 = __floats2half2_rn(p[0] * s_a, p[1] * s_a);
      const __half2 h1 = __floats2half2_rn(p[2] * s_b, p[3] * s_b);
      S.zs[0][gr] = fmaf(p[0], z_a, fmaf(p[2], z_b, S.zs[0][gr]));
      S.zs[1][gr] = fmaf(p[1], z_a, fmaf(p[3], z_b, S.zs[1][gr]));
      const uint32_t b0 = movmatrix_t(*(const uint32_t*)&h0);
      const uint32_t b1 = movmatrix_t(*(const uint32_t*)&h1);
      const uint32_t b0a = b0 & mA, b1a = b1 & mA, b0b = b0 & mBB, b1b = b1 & mBB;
#pragma unroll
      for (int jj = 0; jj < MPG; ++jj) {
        const int j = gr * MPG + jj;
        uint32_t a0, a1, a2, a3, c0, c1, c2, c3;
        switch (s) {
          case 0:
            a0 = code_sub<0>(va_w[j][0]); a1 = code_sub<0>(va_w[j][1]); a2 = code_sub<1>(va_w[j][0]); a3 = code_sub<1>(va_w[j][1]);
            c0 = code_sub<0>(vb_w[j][0]); c1 = code_sub<0>(vb_w[j][1]); c2 = code_sub<1>(vb_w[j][0]); c3 = code_sub<1>(vb_w[j][1]);
            break;
          case 1:
            a0 = code_sub<2>(va_w[j][0]); a1 = code_sub<2>(va_w[j][1]); a2 = code_sub<3>(va_w[j][0]); a3 = code_sub<3>(va_w[j][1]);
            c0 = code_sub<2>(vb_w[j][0]); c1 = code_sub<2>(vb_w[j][1]); c2 = code_sub<3>(vb_w[j][0]); c3 = code_sub<3>(vb_w[j][1]);
            break;
          case 2:
            a0 = code_sub<4>(va_w[j][0]); a1 = code_sub<4>(va_w[j][1]); a2 = code_sub<5>(va_w[j][0]); a3 = code_sub<5>(va_w[j][1]);
            c0 = code_sub<4>(vb_w[j][0]); c1 = code_sub<4>(vb_w[j][1]); c2 = code_sub<5>(vb_w[j][0]); c3 = code_sub<5>(vb_w[j][1]);
            break;
          default:
            a0 = code_sub<6>(va_w[j][0]); a1 = code_sub<6>(va_w[j][1]); a2 = code_sub<7>(va_w[j][0]); a3 = code_sub<7>(va_w[j][1]);
            c0 = code_sub<6>(vb_w[j][0]); c1 = code_sub<6>(vb_w[j][1]); c2 = code_sub<7>(vb_w[j][0]); c3 = code_sub<7>(vb_w[j][1]);
            break;
        }
        mma_f16(S.oacc[j], a0, a1, a2, a3, b0a, b1a);
        mma_f16(S.oacc[j], c0, c1, c2, c3, b0b, b1b);
      }
    }
  }
}

// Merge the two streams of each head (columns n and n + 4 live in lanes tq and
// tq ^ 2) into the lanes with tq < 2, after l, bs and zs were summed over the
// gid lanes.  Stream states start at m = -1e30, so an empty stream has weight 0.
template <int NG>
__device__ __forceinline__ void merge_pair_streams(Int2State<NG>& S) {
#pragma unroll
  for (int hc = 0; hc < 2; ++hc) {
    const float mo = __shfl_xor_sync(0xffffffffu, S.m[hc], 2);
    const float M = fmaxf(S.m[hc], mo);
    const float fa = ex2(S.m[hc] - M), fb = ex2(mo - M);
    S.m[hc] = M;
    S.l[hc] = S.l[hc] * fa + __shfl_xor_sync(0xffffffffu, S.l[hc], 2) * fb;
#pragma unroll
    for (int gr = 0; gr < NG; ++gr) {
      S.zs[hc][gr] = S.zs[hc][gr] * fa + __shfl_xor_sync(0xffffffffu, S.zs[hc][gr], 2) * fb;
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      S.oacc[j][hc] = S.oacc[j][hc] * fa + __shfl_xor_sync(0xffffffffu, S.oacc[j][hc], 2) * fb;
      S.oacc[j][hc + 2] = S.oacc[j][hc + 2] * fa + __shfl_xor_sync(0xffffffffu, S.oacc[j][hc + 2], 2) * fb;
    }
  }
}

// Combine the CTA's warp results (wm, wl, wo) into partial record `slot`.
__device__ __forceinline__ void cta_combine_write(const DecodeArgs& a, const float* wm,
                                                 const float* wl, const float* wo, int slot) {
  const int c = threadIdx.x;  // DEC_NW * 32 == 128 threads, one channel each
  const int G = a.cv.G;
  for (int n = 0; n < G; ++n) {
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < DEC_NW; ++w) M = fmaxf(M, wm[w * MAX_G + n]);
    float Ls = 0.f, O = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < DEC_NW; ++w) {
        const float mw = wm[w * MAX_G + n];
        const float f = mw == -INFINITY ? 0.f : ex2(mw - M);
        Ls = fmaf(wl[w * MAX_G + n], f, Ls);
        O = fmaf(wo[(w * MAX_G + n) * D + c], f, O);
      }
    }
    float* rec = a.part + ((size_t)slot * G + n) * PART_STRIDE;
    if (c == 0) {
      rec[0] = M;
      rec[1] = Ls;
    }
    rec[PART_O + c] = O;
  }
}


}  // namespace oscar
