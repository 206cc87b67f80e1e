// BF16 window attention on mma.sync tiles, shared by the decode kernels
// (sm_103a): 16-token tiles of BF16 keys/values read straight from global
// memory, QK^T and SV on bf16 tensor-core fragments, online softmax per
// column head.  The sink and recent window are kept in BF16 and attended
// unrotated [News "Together AI 开源 OSCAR…", section "服务系统：混合精度缓存布局";
// Blog "超越TurboQuant…", pipeline paragraph: a BF16 kernel handles sink/recent].
#pragma once

#include "oscar_internal.cuh"

namespace oscar {

// ------------------------------------------------------ BF16 chunk (mma)
struct Bf16State {
  float oacc[8][4];  // o^T: m-tile j rows channel 16gid+2j / 16gid+2j+1, cols heads 2tq, 2tq+1
  float m[2];
  float l[2];
  uint32_t bq[8][2];  // raw q (bf16) B fragments, column = head gid
};

__device__ __forceinline__ uint4 ldg_nc(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// One 16-token tile of BF16 keys/values in registers: the rows this thread
// feeds to the tensor cores.
struct Bf16Tile {
  uint4 ka[4], kb[4];  // K rows 16s+gid and 16s+gid+8, channels 32tq..32tq+31
  uint4 vv[4][2];      // V rows of tokens 16s+{2tq, 2tq+1, 2tq+8, 2tq+9}, channels 16gid..16gid+15
};

__device__ __forceinline__ void bf16_tile_load(Bf16Tile& T, const __nv_bfloat16* Kb,
                                               const __nv_bfloat16* Vb, uint64_t valid, int s,
                                               int gid, int tq) {
  const int ta = 16 * s + gid, tb = ta + 8;
#pragma unroll
  for (int qd = 0; qd < 4; ++qd) {
    T.ka[qd] = ldg_nc(Kb + ta * D + 32 * tq + 8 * qd);
    T.kb[qd] = ldg_nc(Kb + tb * D + 32 * tq + 8 * qd);
  }
  const int t0 = 16 * s + 2 * tq, t2 = t0 + 8;
  const int tk[4] = {t0, t0 + 1, t2, t2 + 1};
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const bool ok = (valid >> tk[u]) & 1;
    const __nv_bfloat16* src = Vb + tk[u] * D + 16 * gid;
    T.vv[u][0] = ok ? ldg_nc(src) : make_uint4(0, 0, 0, 0);
    T.vv[u][1] = ok ? ldg_nc(src + 8) : make_uint4(0, 0, 0, 0);
  }
}

__device__ __forceinline__ void bf16_tile_compute(Bf16State& S, const Bf16Tile& T, uint64_t valid,
                                                  int s, int gid) {
  const float cst = LOG2E * INV_SQRT_D;
  const int ta = 16 * s + gid, tb = ta + 8;
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    const uint4& xa = T.ka[kk >> 1];
    const uint4& xb = T.kb[kk >> 1];
    const uint32_t a0 = (kk & 1) ? xa.z : xa.x, a2 = (kk & 1) ? xa.w : xa.y;
    const uint32_t a1 = (kk & 1) ? xb.z : xb.x, a3 = (kk & 1) ? xb.w : xb.y;
    mma_bf16(acc, a0, a1, a2, a3, S.bq[kk][0], S.bq[kk][1]);
  }
  const bool va = (valid >> ta) & 1, vb = (valid >> tb) & 1;
  float lam[4];
  lam[0] = va ? acc[0] * cst : -INFINITY;
  lam[1] = va ? acc[1] * cst : -INFINITY;
  lam[2] = vb ? acc[2] * cst : -INFINITY;
  lam[3] = vb ? acc[3] * cst : -INFINITY;
#pragma unroll
  for (int hc = 0; hc < 2; ++hc) {
    float pm = fmaxf(lam[hc], lam[hc + 2]);
    pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, 4));
    pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, 8));
    pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, 16));
    const float mn = fmaxf(S.m[hc], pm);
    if (mn > S.m[hc]) {  // rescale only when the running max moves
      const float al = ex2(S.m[hc] - mn);
      S.m[hc] = mn;
      S.l[hc] *= al;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        S.oacc[j][hc] *= al;
        S.oacc[j][hc + 2] *= al;
      }
    }
  }
  float p[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) p[e] = ex2(lam[e] - S.m[e & 1]);
  const __nv_bfloat162 h0 = __floats2bfloat162_rn(p[0], p[1]);
  const __nv_bfloat162 h1 = __floats2bfloat162_rn(p[2], p[3]);
  const float2 f0 = __bfloat1622float2(h0), f1 = __bfloat1622float2(h1);
  S.l[0] += f0.x + f1.x;
  S.l[1] += f0.y + f1.y;
  const uint32_t b0 = movmatrix_t(*(const uint32_t*)&h0);
  const uint32_t b1 = movmatrix_t(*(const uint32_t*)&h1);
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const uint32_t x0 = ((const uint32_t*)&T.vv[0][j >> 2])[j & 3];
    const uint32_t x1 = ((const uint32_t*)&T.vv[1][j >> 2])[j & 3];
    const uint32_t x2 = ((const uint32_t*)&T.vv[2][j >> 2])[j & 3];
    const uint32_t x3 = ((const uint32_t*)&T.vv[3][j >> 2])[j & 3];
    mma_bf16(S.oacc[j], prmt(x0, x1, 0x5410), prmt(x0, x1, 0x7632), prmt(x2, x3, 0x5410),
             prmt(x2, x3, 0x7632), b0, b1);
  }
}

// Tiles s0 .. s0+ns-1 (16 tokens each) of 64 BF16 keys/values, row-major
// [64][128] at Kb / Vb; token t is used iff bit t of `valid` is set.  With DB
// the next tile's loads are in flight while the current one is computed (more
// registers); without, tiles are loaded one at a time.
template <bool DB>
__device__ __forceinline__ void bf16_span_mma(Bf16State& S, const __nv_bfloat16* Kb,
                                              const __nv_bfloat16* Vb, uint64_t valid, int lane,
                                              int s0, int ns) {
  const int gid = lane >> 2, tq = lane & 3;
  if (DB) {
    Bf16Tile A, Bt;
    bf16_tile_load(A, Kb, Vb, valid, s0, gid, tq);
    for (int s = s0; s < s0 + ns; s += 2) {
      if (s + 1 < s0 + ns) bf16_tile_load(Bt, Kb, Vb, valid, s + 1, gid, tq);
      if ((valid >> (16 * s)) & 0xFFFFull) bf16_tile_compute(S, A, valid, s, gid);
      if (s + 2 < s0 + ns) bf16_tile_load(A, Kb, Vb, valid, s + 2, gid, tq);
      if (s + 1 < s0 + ns && ((valid >> (16 * (s + 1))) & 0xFFFFull))
        bf16_tile_compute(S, Bt, valid, s + 1, gid);
    }
  } else {
    for (int s = s0; s < s0 + ns; ++s) {
      if (!((valid >> (16 * s)) & 0xFFFFull)) continue;
      Bf16Tile A;
      bf16_tile_load(A, Kb, Vb, valid, s, gid, tq);
      bf16_tile_compute(S, A, valid, s, gid);
    }
  }
}

template <bool DB>
__device__ __forceinline__ void bf16_chunk_mma(Bf16State& S, const __nv_bfloat16* Kb,
                                               const __nv_bfloat16* Vb, uint64_t valid, int lane) {
  bf16_span_mma<DB>(S, Kb, Vb, valid, lane, 0, 4);
}


}  // namespace oscar

