// Decode attention over the three-region INT2 KV cache (sm_103a).
//
// Follows the decode paragraph under the pipeline figure "从离线校准到在线推理的
// pipeline" of "超越TurboQuant：Together AI把2-bit KV Cache推向真实服务": the INT2
// segment is unpacked, dequantised with its scale / zero point and accumulated
// in floating point; the BF16 sink/recent segment is handled separately; the
// parts are merged by online softmax.  Keys and values of the history live in
// the rotated basis x' = x·R [News "Together AI 开源 OSCAR…", section "OSCAR 的
// 不同之处"], so the query is rotated by R_K first and the history output is
// un-rotated by R_V^T before the final merge.
//
// Kernels (one stream, in order):
//   prep_kernel    q' = q·U_K·H·P_br for every query head, packed as the fp16
//                  B operand of the tensor-core QK^T plus per-head logit
//                  constants; resets the work and merge counters
//   decode_kernel  persistent split-K, launched as a programmatic dependent of
//                  prep_kernel: each CTA starts fetching its first pages before
//                  waiting for q'.  Work items are (request, kv head, S pages)
//                  of history or one BF16 window per (request, kv head); each
//                  item writes an online-softmax partial, and the last CTA to
//                  finish an item of a (request, kv head) merges its partials,
//                  un-rotates the history part by R_V^T and writes the output.
#include "oscar_internal.cuh"
#include "oscar_window.cuh"
#include "oscar_pagemath.cuh"

namespace oscar {

namespace {

constexpr int NW = 4;     // warps per decode CTA
constexpr int DEPTH = 4;  // bulk-copy stages per warp

// final merge (merge_kernel)
constexpr int YST = 136;      // fp16 row stride of the mma B operand (conflict-free fragment loads)
constexpr int MERGE_RV_BYTES = RV_FRAG_WORDS * 4;
constexpr int MERGE_Y_BYTES = 2 * MAX_G * YST * 2 > MAX_G * D * 4 ? 2 * MAX_G * YST * 2 : MAX_G * D * 4;


// ------------------------------------------------------------------- prep
// grid (B * Hkv, 4), block 128: one channel quarter per CTA (prep_body).
__global__ void __launch_bounds__(128) prep_kernel(DecodeArgs a) {
  __shared__ PrepSmem sm;
  prep_body(a, blockIdx.x, blockIdx.y, threadIdx.x, sm, true);
}

// ------------------------------------------------------------ smem layout
struct SmemLayout {
  int stage_bytes;   // per stage
  int off_stage, off_mbar, off_qpk, off_qf, off_vs, off_pre, off_red, off_misc, off_cursor, total;
};

// decode_kernel's position in its work list (shared memory, thread 0) and
// the item it hands to the block.
struct DecodeCursor {
  long long lo, hi;        // this CTA's range of positions
  int cb, ck, cc, phase;   // request, kv head, next window chunk, 0 windows / 1 history
  int bl_n, bl_wch;        // CTAs taking part, window chunk weight
  int found, is_win, b, kvh, wc, wch, p0, p1, slot;  // the item
};

// The automatic partition: balanced once the item list would give a CTA more
// than auto_wave_pages() pages (several items per CTA, each paying a start).
__device__ __forceinline__ bool use_balanced(const Sched& sc, int grid, bool bf16_history) {
  return sc.pages > (long long)auto_wave_pages(bf16_history) * grid;
}

// Weight of (b, kvh) in the balanced list: history pages plus wch per
// non-empty window chunk.
__device__ __forceinline__ long long balanced_weight(const int32_t* hl, const int32_t* sl, int b, int wch,
                                                     int* P, unsigned* mask) {
  const int H = hl[b];
  *P = H > 0 ? (H + PAGE - 1) / PAGE : 0;
  *mask = window_chunk_mask(sl[b], H);
  return *P + (long long)wch * __popc(*mask);
}

// Puts the cursor on the segment holding the range's first position.
__device__ inline void cursor_restart(DecodeCursor& c, const long long* pre64, int B, const int32_t* hl,
                                      const int32_t* sl) {
  c.cb = c.lo < c.hi ? balanced_request(pre64, B, c.lo) : B;
  c.ck = 0;
  c.cc = 0;
  if (c.cb < B) {
    int P;
    unsigned mask;
    const long long wb = balanced_weight(hl, sl, c.cb, c.bl_wch, &P, &mask);
    if (wb > 0 && c.lo > pre64[c.cb]) c.ck = (int)((c.lo - pre64[c.cb]) / wb);
  }
}

__device__ inline void cursor_init_balanced(DecodeCursor& c, const Balanced& bl, const long long* pre64, int B,
                                            const int32_t* hl, const int32_t* sl, int cta) {
  c.bl_n = bl.n;
  c.bl_wch = bl.wch;
  c.lo = cta < bl.n ? balanced_lo(bl, cta) : 0;
  c.hi = cta < bl.n ? balanced_lo(bl, cta + 1) : 0;
  c.phase = 0;
  cursor_restart(c, pre64, B, hl, sl);
}

struct WindowPtrs {
  const __nv_bfloat16 *sink_k, *sink_v, *ring_k, *ring_v;
};

// L2 prefetch of the BF16 window chunks whose positions lie in the cursor's
// range (all threads; the cursor as cursor_init_balanced left it).
__device__ inline void prefetch_range_windows(const DecodeCursor& c0, const WindowPtrs& w, int B, int Hkv,
                                              const long long* pre64, const int32_t* hl, const int32_t* sl) {
  if (c0.lo >= c0.hi) return;
  int cb = c0.cb, ck = c0.ck;
  for (int guard = 0; guard < 64 && cb < B && pre64[cb] < c0.hi; ++guard) {
    int P;
    unsigned mask;
    const long long wb = balanced_weight(hl, sl, cb, c0.bl_wch, &P, &mask);
    if (wb == 0 || ck >= Hkv) {
      ++cb;
      ck = 0;
      continue;
    }
    const long long seg = pre64[cb] + (long long)ck * wb;
    if (seg >= c0.hi) break;
    const size_t head = (size_t)cb * Hkv + ck;
    for (int ch = 0; ch < WIN_CHUNKS; ++ch) {
      if (!((mask >> ch) & 1u)) continue;
      const long long x = seg + P + (long long)c0.bl_wch * __popc(mask & ((1u << ch) - 1u));
      if (x < c0.lo || x >= c0.hi) continue;
      // 64 tokens x 256 bytes of K and of V: 128 lines each
      const char* kb = (const char*)(ch == 0 ? w.sink_k + head * SINK * D : w.ring_k + (head * RECENT + 64 * (ch - 1)) * D);
      const char* vb = (const char*)(ch == 0 ? w.sink_v + head * SINK * D : w.ring_v + (head * RECENT + 64 * (ch - 1)) * D);
      for (int l = threadIdx.x; l < 128; l += blockDim.x) {
        asm volatile("prefetch.global.L2 [%0];\n" ::"l"(kb + 128 * l));
        asm volatile("prefetch.global.L2 [%0];\n" ::"l"(vb + 128 * l));
      }
    }
    ++ck;
  }
}

__device__ __noinline__ void cursor_next(DecodeCursor& c, int B, int Hkv, const long long* pre64,
                                         const int32_t* hl, const int32_t* sl);

// The balanced partition's start (all threads): the request weights, this
// CTA's range, an L2 prefetch of its window chunks, and its first item.
__device__ __noinline__ void balanced_setup(DecodeCursor& c, int B, int Hkv, int wch, WindowPtrs w,
                                            long long* pre64, const int32_t* hl, const int32_t* sl) {
  const Balanced bl = make_balanced(sl, hl, B, Hkv, wch, gridDim.x, pre64);
  if (threadIdx.x == 0) cursor_init_balanced(c, bl, pre64, B, hl, sl, blockIdx.x);
  __syncthreads();
  // the window chunks of the range are read with plain loads, which queue
  // behind the whole grid's page copies: ask for all of them at once
  prefetch_range_windows(c, w, B, Hkv, pre64, hl, sl);
  __syncthreads();  // the cursor is read before thread 0 moves it
  if (threadIdx.x == 0) cursor_next(c, B, Hkv, pre64, hl, sl);
  __syncthreads();
}

// The next item of the balanced range into c.found / c.is_win / ... (thread 0).
__device__ __noinline__ void cursor_next(DecodeCursor& c, int B, int Hkv, const long long* pre64,
                                         const int32_t* hl, const int32_t* sl) {
  c.found = 0;
  c.is_win = 0;
  c.wc = 0;
  c.p0 = c.p1 = 0;
  for (;;) {
    if (c.cb >= B || pre64[c.cb] >= c.hi) {
      if (c.phase == 1) return;
      c.phase = 1;
      cursor_restart(c, pre64, B, hl, sl);
      continue;
    }
    int P;
    unsigned mask;
    const long long wb = balanced_weight(hl, sl, c.cb, c.bl_wch, &P, &mask);
    if (wb == 0 || c.ck >= Hkv) {
      ++c.cb;
      c.ck = 0;
      c.cc = 0;
      continue;
    }
    const long long seg = pre64[c.cb] + (long long)c.ck * wb;
    if (seg >= c.hi) {
      c.cb = B;
      continue;
    }
    if (c.phase == 0) {
      while (c.cc < WIN_CHUNKS) {
        const int ch = c.cc++;
        if (!((mask >> ch) & 1u)) continue;
        const long long x = seg + P + (long long)c.bl_wch * __popc(mask & ((1u << ch) - 1u));
        if (x >= c.lo && x < c.hi) {
          c.found = 1;
          c.is_win = 1;
          c.b = c.cb;
          c.kvh = c.ck;
          c.wc = ch;
          c.wch = WIN_CHUNKS;
          c.slot = c.bl_n + B * Hkv + WIN_CHUNKS * (c.cb * Hkv + c.ck) + ch;
          return;
        }
      }
      c.cc = 0;
      ++c.ck;
    } else {
      const long long s0 = c.lo > seg ? c.lo : seg, e0 = c.hi < seg + P ? c.hi : seg + P;
      const int kvh = c.ck++;
      if (s0 < e0) {
        c.found = 1;
        c.b = c.cb;
        c.kvh = kvh;
        c.wch = WIN_CHUNKS;
        c.p0 = (int)(s0 - seg);
        c.p1 = (int)(e0 - seg);
        c.slot = (int)blockIdx.x + c.cb * Hkv + kvh;
        return;
      }
    }
  }
}

// impl: 0 tensor-core INT2, 1 CUDA-core INT2, 2 BF16 history (no INT2 pages),
// 3 tensor-core page pairs, 4 tensor-core with a Lloyd-Max codebook
__host__ __device__ inline SmemLayout smem_layout(int head_bytes, int B, int impl, int G) {
  SmemLayout L;
  // BF16 paths read global memory directly; only INT2 pages use stages
  L.stage_bytes = impl == 2 ? 0 : (head_bytes + 127) & ~127;
  int o = 0;
  L.off_stage = o;
  int stage_total = NW * DEPTH * L.stage_bytes;
  // the warp results alias the stages
  const int wo_bytes = NW * MAX_G * D * 4 + 2 * NW * MAX_G * 4;
  if (stage_total < wo_bytes) stage_total = wo_bytes;
  stage_total = (stage_total + 127) & ~127;  // mbarriers that follow need 8-byte alignment
  o += stage_total;
  L.off_mbar = o;
  o += NW * DEPTH * 8;  // pipeline stages
  L.off_qpk = o;        // tensor-core paths: the G packed query records of the item's kv head
  if (impl == 0 || impl == 3) o += G * QPACK_BYTES;
  if (impl == 4) o += G * QPACK_CB_BYTES;
  L.off_qf = o;
  if (impl == 1) o += MAX_G * D * 4 + MAX_G * 4 * 4;  // fp32 q' in K storage order + z weights
  L.off_vs = o;
  if (impl == 1) o += NW * (MAX_G * PAGE + 2 * 4 * PAGE) * 4;  // CUDA-core per-warp p and s/z
  L.off_pre = o;
  o += ((B + 1) * 8 + 15) & ~15;  // int[B + 1], or long long[B + 1] for the balanced partition
  L.off_red = o;
  o += 2 * NW * 4;  // block reductions of the work-list derivation
  L.off_misc = o;
  o += 16;
  L.off_cursor = o;
  o += ((int)sizeof(DecodeCursor) + 15) & ~15;
  L.total = o;
  return L;
}

// ---------------------------------------------- Lloyd-Max codebook pages
// With a codebook a code's level is c0 + alpha*bit0 + beta*bit1 (symmetric
// levels have no bit0*bit1 term), so a page takes two tensor-core products
// per operand instead of one: the low bit planes against q' * alpha (resp.
// p * s * alpha) and the high bit planes against q' * beta / 2 (resp.
// p * s * beta / 2), into the same accumulators.  c0 moves into the logit
// offset (keys) and into the zero-point sums (values).
struct CbExtra {
  uint32_t bq2[8][2];  // q' B fragments of the high bit plane (qb of the record)
  float va, vb, vc0;   // alpha_V, beta_half_V, c0_V
};

// The four A registers of bit plane P for code positions 2q, 2q + 1 (q = 0..3)
// of words x (rows gid) and y (rows gid + 8).
template <int P>
__device__ __forceinline__ void plane_frag(int q, uint32_t x, uint32_t y, uint32_t& a0, uint32_t& a1,
                                           uint32_t& a2, uint32_t& a3) {
  switch (q) {
    case 0: a0 = code_plane_sub<0, P>(x); a1 = code_plane_sub<0, P>(y); a2 = code_plane_sub<1, P>(x); a3 = code_plane_sub<1, P>(y); break;
    case 1: a0 = code_plane_sub<2, P>(x); a1 = code_plane_sub<2, P>(y); a2 = code_plane_sub<3, P>(x); a3 = code_plane_sub<3, P>(y); break;
    case 2: a0 = code_plane_sub<4, P>(x); a1 = code_plane_sub<4, P>(y); a2 = code_plane_sub<5, P>(x); a3 = code_plane_sub<5, P>(y); break;
    default: a0 = code_plane_sub<6, P>(x); a1 = code_plane_sub<6, P>(y); a2 = code_plane_sub<7, P>(x); a3 = code_plane_sub<7, P>(y); break;
  }
}

template <int NG, bool FULL>
__device__ __forceinline__ void int2_page_mma_cb(Int2State<NG>& S, const CbExtra& X, const uint8_t* stage,
                                                 int nv, int lane) {
  const int gid = lane >> 2, tq = lane & 3;
  constexpr int KPG = 8 / NG;
  constexpr int MPG = 8 / NG;
  const uint8_t* kc = stage;
  const uint8_t* vc = stage + 2048;
  const __half2* ksz = (const __half2*)(stage + 4096);
  const __half2* vsz = (const __half2*)(stage + 4096 + PAGE * NG * 4);

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
      plane_frag<0>(kk & 3, xa, xb, a0, a1, a2, a3);
      mma_f16(acc[s][kk / KPG], a0, a1, a2, a3, S.bq[kk][0], S.bq[kk][1]);
      plane_frag<1>(kk & 3, xa, xb, a0, a1, a2, a3);
      mma_f16(acc[s][kk / KPG], a0, a1, a2, a3, X.bq2[kk][0], X.bq2[kk][1]);
    }
  }
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
        v = fmaf(sz.x, fmaf(acc[s][gr][e], S.ka[hc], S.kb[hc][gr]), fmaf(sz.y, S.kg[hc][gr], v));
      }
      lam[s][e] = (FULL || row < nv) ? v : -INFINITY;
    }
  }
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
    const float fa = (float)(1 << (8 - code_exp_rt(2 * s)));
    const float fb = (float)(1 << (8 - code_exp_rt(2 * s + 1)));
#pragma unroll
    for (int gr = 0; gr < NG; ++gr) {
      const float2 sa = __half22float2(vsz[ta * NG + gr]);
      const float2 sb = __half22float2(vsz[tb * NG + gr]);
      const float s_a = va ? sa.x * fa : 0.f, z_a = va ? fmaf(X.vc0, sa.x, sa.y) : 0.f;
      const float s_b = vb ? sb.x * fb : 0.f, z_b = vb ? fmaf(X.vc0, sb.x, sb.y) : 0.f;
      const float sa0 = s_a * X.va, sa1 = s_a * X.vb, sb0 = s_b * X.va, sb1 = s_b * X.vb;
      const __half2 h0 = __floats2half2_rn(p[0] * sa0, p[1] * sa0);
      const __half2 h1 = __floats2half2_rn(p[2] * sb0, p[3] * sb0);
      const __half2 g0 = __floats2half2_rn(p[0] * sa1, p[1] * sa1);
      const __half2 g1 = __floats2half2_rn(p[2] * sb1, p[3] * sb1);
      S.zs[0][gr] = fmaf(p[0], z_a, fmaf(p[2], z_b, S.zs[0][gr]));
      S.zs[1][gr] = fmaf(p[1], z_a, fmaf(p[3], z_b, S.zs[1][gr]));
      const uint32_t b0 = movmatrix_t(*(const uint32_t*)&h0);
      const uint32_t b1 = movmatrix_t(*(const uint32_t*)&h1);
      const uint32_t c0 = movmatrix_t(*(const uint32_t*)&g0);
      const uint32_t c1 = movmatrix_t(*(const uint32_t*)&g1);
#pragma unroll
      for (int jj = 0; jj < MPG; ++jj) {
        const int j = gr * MPG + jj;
        uint32_t a0, a1, a2, a3;
        plane_frag<0>(s, vw[j][0], vw[j][1], a0, a1, a2, a3);
        mma_f16(S.oacc[j], a0, a1, a2, a3, b0, b1);
        plane_frag<1>(s, vw[j][0], vw[j][1], a0, a1, a2, a3);
        mma_f16(S.oacc[j], a0, a1, a2, a3, c0, c1);
      }
    }
  }
}

// ----------------------------------------------- CUDA-core INT2 page (fp32)
// Lane l scores tokens l and l+32, then accumulates channels 4l..4l+3.
struct CoreState {
  float o[MAX_G][4];
  float m[MAX_G];
  float l[MAX_G];
};

template <int NG>
__device__ __forceinline__ void int2_page_core(CoreState& S, const uint8_t* stage, int nv, int lane,
                                               int G, const float* qst /*[G][128] storage order*/,
                                               const float* kgm /*[MAX_G][4] z weights, log2 units*/,
                                               float* ps /*[G][64]*/,
                                               float* vsz_s /*[2][NG][64]*/) {
  const uint32_t* kc = (const uint32_t*)stage;
  const uint32_t* vc = (const uint32_t*)(stage + 2048);
  const __half2* ksz = (const __half2*)(stage + 4096);
  const __half2* vsz = (const __half2*)(stage + 4096 + PAGE * NG * 4);
  const float cst = LOG2E * INV_SQRT_D;
  float lam[2][MAX_G];
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int t = lane + 32 * r;
    uint32_t w[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) w[k] = kc[t * 8 + k];
    for (int n = 0; n < G; ++n) {
      float acc[NG];
#pragma unroll
      for (int gr = 0; gr < NG; ++gr) acc[gr] = 0.f;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
#pragma unroll
        for (int pos = 0; pos < 16; ++pos) {
          // storage slot (word k, bit 2*pos) holds channel 64A+16B+8C+2D+E with
          // k = 2D+A, pos = 8E+2B+C; its group is channel / g
          const int A = k & 1, B = (pos >> 1) & 3;
          const int gr = NG == 1 ? 0 : NG == 2 ? A : (2 * A + (B >> 1));
          const float code = (float)((w[k] >> (2 * pos)) & 3u);
          acc[gr] = fmaf(code, qst[n * D + k * 16 + pos], acc[gr]);
        }
      }
      float v = 0.f;
#pragma unroll
      for (int gr = 0; gr < NG; ++gr) {
        const float2 sz = __half22float2(ksz[t * NG + gr]);
        v = fmaf(sz.x, acc[gr] * cst, fmaf(sz.y, kgm[n * 4 + gr], v));
      }
      lam[r][n] = t < nv ? v : -INFINITY;
    }
  }
  // V scale / zero of the page into smem (select out invalid tokens)
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int t = lane + 32 * r;
    for (int gr = 0; gr < NG; ++gr) {
      const float2 sz = __half22float2(vsz[t * NG + gr]);
      vsz_s[gr * PAGE + t] = t < nv ? sz.x : 0.f;
      vsz_s[(NG + gr) * PAGE + t] = t < nv ? sz.y : 0.f;
    }
  }
  for (int n = 0; n < G; ++n) {
    float pm = fmaxf(lam[0][n], lam[1][n]);
#pragma unroll
    for (int o = 16; o; o >>= 1) pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, o));
    const float mn = fmaxf(S.m[n], pm);
    const float al = ex2(S.m[n] - mn);
    S.m[n] = mn;
    const float p0 = ex2(lam[0][n] - mn), p1 = ex2(lam[1][n] - mn);
    float ls = p0 + p1;
#pragma unroll
    for (int o = 16; o; o >>= 1) ls += __shfl_xor_sync(0xffffffffu, ls, o);
    S.l[n] = S.l[n] * al + ls;
#pragma unroll
    for (int c = 0; c < 4; ++c) S.o[n][c] *= al;
    ps[n * PAGE + lane] = p0;
    ps[n * PAGE + lane + 32] = p1;
  }
  __syncwarp();
  // channels 4*lane .. 4*lane+3 (one group)
  const int gr = (4 * lane) / (D / NG);
  uint32_t rows[4][4];
#pragma unroll
  for (int c = 0; c < 4; ++c)
#pragma unroll
    for (int k = 0; k < 4; ++k) rows[c][k] = vc[(4 * lane + c) * 4 + k];
  for (int t = 0; t < PAGE; ++t) {
    const int wsel = v_word(t), sh = v_bit(t);
    const float s = vsz_s[gr * PAGE + t], z = vsz_s[(NG + gr) * PAGE + t];
    float vh[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      uint32_t word = rows[c][0];
      word = wsel == 1 ? rows[c][1] : word;
      word = wsel == 2 ? rows[c][2] : word;
      word = wsel == 3 ? rows[c][3] : word;
      vh[c] = fmaf((float)((word >> sh) & 3u), s, z);
    }
    for (int n = 0; n < G; ++n) {
      const float p = ps[n * PAGE + t];
#pragma unroll
      for (int c = 0; c < 4; ++c) S.o[n][c] = fmaf(p, vh[c], S.o[n][c]);
    }
  }
  __syncwarp();
}

// Page ids of a warp's pages k = 0, 1, ... (page p0 + warp + k*NW of request
// b), held 32 at a time in registers (lane i keeps page 32*blk + i) so that
// no page waits on a dependent page-table load.
struct PageIds {
  int cur, a, b;
};

__device__ __forceinline__ int page_id_load(const CacheView& cv, int b, int first, int k, int n) {
  return k < n ? __ldg(cv.page_table + (size_t)b * cv.max_pages_per_req + first + k * NW) : -1;
}

__device__ __forceinline__ void page_ids_init(PageIds& P, const CacheView& cv, int b, int first, int n,
                                              int lane) {
  P.cur = 0;
  P.a = page_id_load(cv, b, first, lane, n);
  P.b = page_id_load(cv, b, first, 32 + lane, n);
}

// All lanes call; k must lie in the current block or the next one.
__device__ __forceinline__ int page_id_at(const PageIds& P, int k) {
  const int v = ((k >> 5) == P.cur) ? P.a : P.b;
  return __shfl_sync(0xffffffffu, v, k & 31);
}

// Call when page k (k % 32 == 0, k > 0) is reached.
__device__ __forceinline__ void page_ids_advance(PageIds& P, const CacheView& cv, int b, int first,
                                                 int n, int lane) {
  P.a = P.b;
  ++P.cur;
  P.b = page_id_load(cv, b, first, 32 * (P.cur + 1) + lane, n);
}

// ----------------------------------------------------------------- decode
__device__ __forceinline__ float4 fma4(float4 o, float w, float4 acc) {
  acc.x = fmaf(o.x, w, acc.x);
  acc.y = fmaf(o.y, w, acc.y);
  acc.z = fmaf(o.z, w, acc.z);
  acc.w = fmaf(o.w, w, acc.w);
  return acc;
}

__device__ __forceinline__ float4 scale4(float4 o, float w) {
  return make_float4(o.x * w, o.y * w, o.z * w, o.w * w);
}

__device__ __forceinline__ uint32_t split_hi(float a, float b, uint32_t* lo) {
  const __half ha = __float2half_rn(a), hb = __float2half_rn(b);
  const __half la = __float2half_rn(a - __half2float(ha)), lb = __float2half_rn(b - __half2float(hb));
  *lo = (uint32_t)__half_as_ushort(la) | ((uint32_t)__half_as_ushort(lb) << 16);
  return (uint32_t)__half_as_ushort(ha) | ((uint32_t)__half_as_ushort(hb) << 16);
}

// ------------------------------------------------------------------ merge
// grid = B * Hkv * (G / hpc), block = MW * 32, launched as a programmatic
// dependent of decode_kernel.  CTA (b, kvh, head group) merges the partial
// records of query heads h0 .. h0 + hpc - 1 of request b, kv head kvh [Blog,
// pipeline paragraph: the INT2 and BF16 parts are combined by online
// softmax].  A merge reads every partial record of its heads once, so small
// batches spread it over more CTAs (hpc < G) to use more SMs' load bandwidth:
//   * before waiting for the decode kernel it derives the work list (the same
//     one the decode kernel used) and starts a bulk copy of the R_V fragments
//     (64 KB) into shared memory;
//   * the MW / hpc warps of head n's team take every (MW / hpc)-th record of the
//     list (history partials, then window partials) and LSE-merge history and
//     window separately, with all of their loads in one round (each lane
//     holds channels 4*lane .. 4*lane+3);
//   * warp n combines its team into (M, L, O'), normalises O'/L and writes it
//     as fp16 high and low parts; o = (O'/L)·R_V^T is three fp16 products per
//     tile (hi·hi, hi·lo, lo·hi) with fp32 accumulation, warp w < 8 owning
//     output channels 16w .. 16w+15;
//   * warp n writes head n's LSE-merge of history and window.
constexpr int MW = 16;       // warps of the merge kernel
constexpr int MERGE_MQ = 4;   // records per warp and round of loads

struct MergeLayout {
  int off_rv, off_y, off_tm, off_to, off_win, off_wo, off_h, off_mbar, off_red, off_pre, total;
};

__host__ __device__ inline MergeLayout merge_layout(int B) {
  MergeLayout L;
  int o = 0;
  L.off_rv = o;
  o += MERGE_RV_BYTES;
  L.off_y = o;
  o += MERGE_Y_BYTES;
  L.off_tm = o;               // team m, l of history and window: [4][MW]
  o += 4 * MW * 4;
  L.off_to = o;               // team o of history and window: [2][MW][128]
  o += 2 * MW * D * 4;
  L.off_win = o;              // window m, l: [2][MAX_G]
  o += 2 * MAX_G * 4;
  L.off_wo = o;               // window o: [MAX_G][128]
  o += MAX_G * D * 4;
  L.off_h = o;                // history M, L, fp16 scale: [3][MAX_G]
  o += 3 * MAX_G * 4 + 8;
  L.off_mbar = (o + 7) & ~7;
  o = L.off_mbar + 16;
  L.off_red = o;
  o += 64 * 4;
  L.off_pre = (o + 7) & ~7;
  o = L.off_pre + (((B + 1) * 8 + 15) & ~15);  // int[B + 1], or long long[B + 1] for the balanced list
  L.total = o;
  return L;
}

__global__ void __launch_bounds__(MW * 32) merge_kernel(DecodeArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  const CacheView& cv = a.cv;
  const int G = cv.G, Hkv = cv.Hkv, t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const int gid = lane >> 2, tq = lane & 3;
  const int HPC = a.merge_hpc, NHG = G / HPC;
  const int h0 = (blockIdx.x % NHG) * HPC;
  const int b = (blockIdx.x / NHG) / Hkv, kvh = (blockIdx.x / NHG) % Hkv;
  const MergeLayout ML = merge_layout(a.B);
  const uint4* Rf = (const uint4*)(smem + ML.off_rv);
  uint32_t* yh = (uint32_t*)(smem + ML.off_y);  // [MAX_G][YST] fp16 high parts
  uint32_t* yl = yh + MAX_G * YST / 2;          // [MAX_G][YST] fp16 low parts
  float* yo = (float*)(smem + ML.off_y);        // [MAX_G][128] history output (aliases yh, yl)
  float* tm = (float*)(smem + ML.off_tm);
  float* tl = tm + MW;
  float* to = (float*)(smem + ML.off_to);
  float* wmv = (float*)(smem + ML.off_win);
  float* wlv = wmv + MAX_G;
  float* wov = (float*)(smem + ML.off_wo);
  float* hM = (float*)(smem + ML.off_h);
  float* hL = hM + MAX_G;
  float* ysc = hL + MAX_G;
  uint64_t* mbar = (uint64_t*)(smem + ML.off_mbar);
  int* red = (int*)(smem + ML.off_red);
  int* pre = (int*)(smem + ML.off_pre);
  const bool unrot = !a.bf16_history && a.rot.mode != OSCAR_ROT_NONE;
  pdl_launch_dependents();  // the next stream work waits for this grid before it reads
  if (t == 0) mbar_init(mbar, 1);
  fence_proxy_async();
  __syncthreads();
  if (unrot && t == 0) {
    mbar_expect_tx(mbar, MERGE_RV_BYTES);
    bulk_g2s(smem + ML.off_rv, a.rot.RV_frag + (size_t)kvh * RV_FRAG_WORDS, MERGE_RV_BYTES, mbar);
  }
  // history lengths come from earlier stream work: the work list can be
  // derived before the wait
  const int32_t* hl = a.step_pred ? a.pred + a.B : cv.hist_lens;  // as the decode kernel's
  const int32_t* sl = a.step_pred ? a.pred : cv.seq_lens;
  int nb, base, wslot, wch;
  unsigned wmask;  // window records that exist
  long long* pre64 = (long long*)(smem + ML.off_pre);
  const int unit = a.bf16_history ? BF16_HEAD_BYTES : cv.head_bytes;
  bool bal = a.balanced == 1;
  Sched sc;
  if (!bal) {
    sc = make_sched(hl, a.B, Hkv, a.target_items, a.resident, unit, pre, red, pages_granule(a.impl),
                    auto_wave_pages(a.bf16_history));
    bal = a.balanced == 2 && use_balanced(sc, a.bal_grid, a.bf16_history);  // as decode_kernel decides
  }
  if (bal) {
    const Balanced bl = make_balanced(sl, hl, a.B, Hkv, a.bal_wch, a.bal_grid, pre64);
    // the balanced partition's list: the history records of the CTAs owning
    // this segment's pages, then one record per non-empty window chunk
    const int H = hl[b], Lq = sl[b];
    const int P = H > 0 ? (H + PAGE - 1) / PAGE : 0;
    wmask = window_chunk_mask(Lq, H);
    const long long seg = pre64[b] + (long long)kvh * (P + bl.wch * __popc(wmask));
    nb = 0;
    base = 0;
    if (P > 0) {
      const int i0 = balanced_owner(bl, seg), i1 = balanced_owner(bl, seg + P - 1);
      nb = i1 - i0 + 1;
      base = i0 + b * Hkv + kvh;
    }
    wch = WIN_CHUNKS;
    wslot = bl.n + a.B * Hkv + WIN_CHUNKS * (b * Hkv + kvh);
  } else {
    const int pages_b = (hl[b] + PAGE - 1) / PAGE;
    nb = (pages_b + sc.S - 1) / sc.S;
    base = pre[b] + kvh * nb;
    wch = sc.wch;
    wslot = sc.n_hist + (b * Hkv + kvh) * sc.wch;
    wmask = (1u << wch) - 1u;
  }
  const int WPH = MW / HPC;  // warps per head
  const int n = warp / WPH, r = warp % WPH;  // head h0 + n of the kv group
  if (n < HPC && lane == 0 && r < nb + wch) {
    // warm the address translation of this warp's records while the decode
    // kernel finishes (the line is written again before it is read)
    const int slot = r < nb ? base + r : wslot + (r - nb);
    asm volatile("prefetch.global.L2 [%0];\n" ::"l"(a.part + ((size_t)slot * G + h0 + n) * PART_STRIDE));
  }
  pdl_wait();  // the decode kernel's partial records are complete and visible
  if (a.step_pred && t == 0 && kvh == 0 && h0 == 0) {
    // decode step: the request's new lengths (the step kernel's append left
    // them to this kernel, which runs once every reader of the old ones is done)
    cv.seq_lens[b] = a.pred[b];
    cv.hist_lens[b] = a.pred[a.B + b];
  }

  // ---- team member: records q = r, r + WPH, ... of the list (history
  // partials 0..nb-1, then window partials nb..nb+wch-1)
  float* tmw = tl + MW;
  float* tlw = tmw + MW;
  float* tow = to + MW * D;
  if (n < HPC) {
    float M = -INFINITY, Ls = 0.f, Mw = -INFINITY, Lw = 0.f;
    float4 O = make_float4(0.f, 0.f, 0.f, 0.f), OW = O;
    const int nrec = nb + wch;
    for (int q0 = r; q0 < nrec; q0 += WPH * MERGE_MQ) {
      float mq[MERGE_MQ], lq[MERGE_MQ];
      float4 oq[MERGE_MQ];
#pragma unroll
      for (int u = 0; u < MERGE_MQ; ++u) {
        const int q = q0 + u * WPH;
        const bool have = q < nb || (q < nrec && ((wmask >> (q - nb)) & 1u));
        const int slot = q < nb ? base + q : wslot + (q - nb);
        const float* rec = a.part + ((size_t)(have ? slot : 0) * G + h0 + n) * PART_STRIDE;
        mq[u] = have ? __ldcg(rec) : -INFINITY;
        lq[u] = have ? __ldcg(rec + 1) : 0.f;
        oq[u] = have ? __ldcg((const float4*)(rec + PART_O) + lane) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
      float mx = M, mxw = Mw;
#pragma unroll
      for (int u = 0; u < MERGE_MQ; ++u) {
        const bool hist = q0 + u * WPH < nb;
        if (lq[u] > 0.f) {
          if (hist) mx = fmaxf(mx, mq[u]);
          else mxw = fmaxf(mxw, mq[u]);
        }
      }
      const float f = (M == -INFINITY || mx == -INFINITY) ? 0.f : ex2(M - mx);
      const float fw = (Mw == -INFINITY || mxw == -INFINITY) ? 0.f : ex2(Mw - mxw);
      Ls *= f;
      O = scale4(O, f);
      Lw *= fw;
      OW = scale4(OW, fw);
      M = mx;
      Mw = mxw;
#pragma unroll
      for (int u = 0; u < MERGE_MQ; ++u) {
        const bool hist = q0 + u * WPH < nb;
        const float w = lq[u] > 0.f ? ex2(mq[u] - (hist ? M : Mw)) : 0.f;
        if (hist) {
          Ls = fmaf(lq[u], w, Ls);
          O = fma4(oq[u], w, O);
        } else {
          Lw = fmaf(lq[u], w, Lw);
          OW = fma4(oq[u], w, OW);
        }
      }
    }
    if (lane == 0) {
      tm[warp] = M;
      tl[warp] = Ls;
      tmw[warp] = Mw;
      tlw[warp] = Lw;
    }
    ((float4*)(to + warp * D))[lane] = O;
    ((float4*)(tow + warp * D))[lane] = OW;
  }
  __syncthreads();
  // ---- warp n: head h0 + n's history total, normalised and scaled for the fp16 split
  if (warp < HPC) {
    const int h = warp;
    // team member k's m and l in lane k
    const float lk = lane < WPH ? tl[h * WPH + lane] : 0.f;
    const float mk = lane < WPH ? tm[h * WPH + lane] : -INFINITY;
    const float lwk = lane < WPH ? tlw[h * WPH + lane] : 0.f;
    const float mwk = lane < WPH ? tmw[h * WPH + lane] : -INFINITY;
    float M = lk > 0.f ? mk : -INFINITY, Mw = lwk > 0.f ? mwk : -INFINITY;
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
      Mw = fmaxf(Mw, __shfl_xor_sync(0xffffffffu, Mw, o));
    }
    const float wk = lk > 0.f ? ex2(mk - M) : 0.f;
    const float wwk = lwk > 0.f ? ex2(mwk - Mw) : 0.f;
    float Ls = lk * wk, Lw = lwk * wwk;
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      Ls += __shfl_xor_sync(0xffffffffu, Ls, o);
      Lw += __shfl_xor_sync(0xffffffffu, Lw, o);
    }
    float4 O = make_float4(0.f, 0.f, 0.f, 0.f), OW = O;
#pragma unroll
    for (int k = 0; k < MW; ++k) {
      const float w = __shfl_sync(0xffffffffu, wk, k), ww = __shfl_sync(0xffffffffu, wwk, k);
      if (k < WPH) {
        O = fma4(((const float4*)(to + (h * WPH + k) * D))[lane], w, O);
        OW = fma4(((const float4*)(tow + (h * WPH + k) * D))[lane], ww, OW);
      }
    }
    if (lane == 0) {
      wmv[h] = Mw;
      wlv[h] = Lw;
    }
    ((float4*)(wov + h * D))[lane] = OW;
    const float4 Y = scale4(O, Ls > 0.f ? 1.f / Ls : 0.f);
    float am = fmaxf(fmaxf(fabsf(Y.x), fabsf(Y.y)), fmaxf(fabsf(Y.z), fabsf(Y.w)));
#pragma unroll
    for (int o = 16; o; o >>= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
    // up = 2^(12 - ex) (at most 2^100), ex the frexp exponent of am, from its exponent bits
    const int ex = (int)((__float_as_uint(am) >> 23) & 0xffu) - 126;
    const float up = am > 0.f ? pow2i(min(12 - ex, 100)) : 1.f;
    if (lane == 0) {
      hM[h] = Ls > 0.f ? M : -INFINITY;
      hL[h] = Ls;
      ysc[h] = up;
    }
    if (unrot) {
      uint32_t l0, l1;
      const uint32_t h0 = split_hi(Y.x * up, Y.y * up, &l0);
      const uint32_t h1 = split_hi(Y.z * up, Y.w * up, &l1);
      *(uint2*)(yh + h * (YST / 2) + 2 * lane) = make_uint2(h0, h1);
      *(uint2*)(yl + h * (YST / 2) + 2 * lane) = make_uint2(l0, l1);
    } else {
      ((float4*)(yo + h * D))[lane] = scale4(Y, up);
    }
  } else if (unrot && warp < MAX_G) {
    // B operand rows of absent heads are 0
    *(uint2*)(yh + warp * (YST / 2) + 2 * lane) = make_uint2(0u, 0u);
    *(uint2*)(yl + warp * (YST / 2) + 2 * lane) = make_uint2(0u, 0u);
  }
  __syncthreads();
  if (unrot) {
    if (!mbar_wait(mbar, 0)) record_error(cv.err, OSCAR_ERR_TIMEOUT);
    float d[4] = {0.f, 0.f, 0.f, 0.f};
    if (warp < 8) {
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const uint32_t bh0 = yh[gid * (YST / 2) + 8 * ks + tq], bh1 = yh[gid * (YST / 2) + 8 * ks + 4 + tq];
        const uint32_t bl0 = yl[gid * (YST / 2) + 8 * ks + tq], bl1 = yl[gid * (YST / 2) + 8 * ks + 4 + tq];
        const uint4 ah = Rf[rv_frag_index(0, warp, ks, lane) / 4];
        const uint4 al = Rf[rv_frag_index(1, warp, ks, lane) / 4];
        mma_f16(d, ah.x, ah.y, ah.z, ah.w, bh0, bh1);
        mma_f16(d, ah.x, ah.y, ah.z, ah.w, bl0, bl1);
        mma_f16(d, al.x, al.y, al.z, al.w, bh0, bh1);
      }
    }
    __syncthreads();  // B operands consumed: yo may overwrite them
    if (warp < 8) {
      const int c = 16 * warp + gid;
      yo[(2 * tq) * D + c] = d[0];
      yo[(2 * tq + 1) * D + c] = d[1];
      yo[(2 * tq) * D + c + 8] = d[2];
      yo[(2 * tq + 1) * D + c + 8] = d[3];
    }
    __syncthreads();
  }
  // ---- warp n: LSE-merge of history and window for head h0 + n
  if (warp < HPC) {
    const int h = warp;
    const float M = hM[h], Ls = hL[h], mw = wmv[h], lw = wlv[h];
    const float down = 1.f / ysc[h];
    const float4 Oh = ((const float4*)(yo + h * D))[lane];
    const float4 Ow = ((const float4*)(wov + h * D))[lane];
    const float M2 = fmaxf(Ls > 0.f ? M : -INFINITY, lw > 0.f ? mw : -INFINITY);
    float o[4] = {0.f, 0.f, 0.f, 0.f};
    float lse = -INFINITY;
    if (M2 != -INFINITY) {
      const float fh = Ls > 0.f ? ex2(M - M2) : 0.f;
      const float fw = lw > 0.f ? ex2(mw - M2) : 0.f;
      const float den = Ls * fh + lw * fw;
      const float inv = 1.f / den;
      const float hw = Ls * fh * down;  // the history output is normalised and scaled by ysc
      o[0] = fmaf(Oh.x, hw, Ow.x * fw) * inv;
      o[1] = fmaf(Oh.y, hw, Ow.y * fw) * inv;
      o[2] = fmaf(Oh.z, hw, Ow.z * fw) * inv;
      o[3] = fmaf(Oh.w, hw, Ow.w * fw) * inv;
      lse = (M2 + log2f(den)) * LN2;
    }
    const size_t row = (size_t)b * cv.Hq + kvh * G + h0 + h;
    __nv_bfloat162 o01 = __floats2bfloat162_rn(o[0], o[1]);
    __nv_bfloat162 o23 = __floats2bfloat162_rn(o[2], o[3]);
    uint2 pk;
    pk.x = *(const uint32_t*)&o01;
    pk.y = *(const uint32_t*)&o23;
    *(uint2*)(a.out + row * D + 4 * lane) = pk;
    if (a.lse && lane == 0) a.lse[row] = lse;
  }
}

// IMPL: 0 INT2 history on tensor cores, 1 INT2 history on CUDA cores,
// 2 BF16 history (the baseline; no INT2 code, double-buffered BF16 tiles).
template <int NG, int IMPL>
// Three CTAs per SM fit the shared memory of g = 128 pages only (4608-byte
// stages); at g = 64 and 32 two do, and the register budget follows.
__global__ void __launch_bounds__(NW * 32, (NG == 1 && (IMPL == 0 || IMPL == 3 || IMPL == 4)) ? 3 : 2)
    decode_kernel(DecodeArgs a) {
  constexpr bool BF16H = (IMPL == 2);
  extern __shared__ __align__(128) uint8_t smem[];
  const CacheView& cv = a.cv;
  const SmemLayout L = smem_layout(cv.head_bytes, a.B, IMPL, cv.G);
  uint64_t* mbar = (uint64_t*)(smem + L.off_mbar);
  float* qf = (float*)(smem + L.off_qf);  // CUDA-core path: [MAX_G][D] q' + [MAX_G][4] z weights
  float* vsw = (float*)(smem + L.off_vs);
  int* pre = (int*)(smem + L.off_pre);
  int* red = (int*)(smem + L.off_red);
  int* misc = (int*)(smem + L.off_misc);
  float* wm = (float*)(smem + L.off_stage);
  float* wl = wm + NW * MAX_G;
  float* wo = wl + NW * MAX_G;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gid = lane >> 2, tq = lane & 3;
  const int G = cv.G, Hkv = cv.Hkv;

  // merge_kernel may be scheduled as CTAs of this grid retire; in a decode
  // step only after this CTA has waited for the step kernel (the merge reads
  // the lengths before its own wait)
  if (!a.step_pred) pdl_launch_dependents();
  if (threadIdx.x < NW * DEPTH) mbar_init(&mbar[threadIdx.x], 1);
  uint8_t* qpk = smem + L.off_qpk;
  if (threadIdx.x == 0) misc[1] = 0;
  fence_proxy_async();
  __syncthreads();

  // history lengths and page tables come from earlier stream work (or, in a
  // decode step, from the step kernel's prediction): readable before the wait
  const int unit = a.bf16_history ? BF16_HEAD_BYTES : cv.head_bytes;
  const int32_t* hl = a.step_pred ? a.pred + a.B : cv.hist_lens;
  const int32_t* sl = a.step_pred ? a.pred : cv.seq_lens;
  auto wait_prev = [&]() {  // the wait for the kernel before, once
    pdl_wait();
    if (a.step_pred) pdl_launch_dependents();
  };
  uint32_t seq = 0;  // stages consumed by this warp so far
  bool waited = false;

  // The work list, one item at a time: a window item is chunk wc of (b,
  // kvh)'s BF16 window (wch == 5: warp w takes its 16 tokens of the chunk;
  // wch == 1: all five chunks, the warps in turn), a history item pages
  // [p0, p1) of (b, kvh); each writes partial record slot.  Thread 0 derives
  // the next item from a cursor kept in shared memory (nothing of it stays
  // in registers across the page loop) and broadcasts it.
  //  * item list: make_sched's items, the first one static (blockIdx.x),
  //    later ones from the work counter;
  //  * balanced: CTA i takes positions [lo_i, lo_i+1) of the list of all
  //    (b, kvh) in order, each weighing its history pages plus bal_wch per
  //    non-empty window chunk; first the window chunks whose position lies
  //    in the range, then the history pages in it.
  // a.balanced == 2 picks the balanced partition when the item list would
  // give a CTA more than one wave's worth of pages (the merge decides alike).
  DecodeCursor* cur = (DecodeCursor*)(smem + L.off_cursor);
  Sched sc;
  bool bal = a.balanced == 1;
  if (!bal) {
    sc = make_sched(hl, a.B, Hkv, a.target_items, a.resident, unit, pre, red, pages_granule(a.impl),
                    auto_wave_pages(a.bf16_history));
    bal = a.balanced == 2 && use_balanced(sc, gridDim.x, a.bf16_history);
  }
  if (bal)  // out of line: the item list's path stays short
    balanced_setup(*cur, a.B, Hkv, a.bal_wch, WindowPtrs{cv.sink_k, cv.sink_v, cv.ring_k, cv.ring_v},
                   (long long*)pre, hl, sl);
  const int total = bal ? 0 : sc.n_hist + sc.n_win;
  int it = blockIdx.x;  // item list: first item static, later ones from the work counter

  for (;;) {
    bool is_win;
    int b, kvh, wc = 0, wch, p0 = 0, p1 = 0, slot;
    if (bal) {
      if (!cur->found) break;
      is_win = cur->is_win;
      b = cur->b;
      kvh = cur->kvh;
      wc = cur->wc;
      wch = cur->wch;
      p0 = cur->p0;
      p1 = cur->p1;
      slot = cur->slot;
    } else {
      if (it >= total) break;
      int idx;
      if (sc.win_first) {
        is_win = it < sc.n_win;
        idx = is_win ? it : it - sc.n_win;
      } else {
        is_win = it >= sc.n_hist;
        idx = is_win ? it - sc.n_hist : it;
      }
      wch = sc.wch;
      if (is_win) {
        b = idx / (Hkv * sc.wch);
        kvh = (idx / sc.wch) % Hkv;
        wc = idx % sc.wch;
        slot = sc.n_hist + idx;
      } else {
        int jj = 0;
        hist_item_coords(idx, pre, a.B, Hkv, hl, sc.S, b, kvh, jj);
        p0 = jj * sc.S;
        p1 = p0 + sc.S;
        slot = idx;
      }
    }
    const int hist_b = hl[b];
    const int pages_b = (hist_b + PAGE - 1) / PAGE;
    if (p1 > pages_b) p1 = pages_b;

    if (is_win || BF16H) {
      // ---------------------------------------------------- BF16 tokens
      if (a.step_pred && !waited) {  // the step kernel writes the window
        wait_prev();
        waited = true;
      }
      Bf16State S;
#pragma unroll
      for (int j = 0; j < 8; ++j) S.oacc[j][0] = S.oacc[j][1] = S.oacc[j][2] = S.oacc[j][3] = 0.f;
      S.m[0] = S.m[1] = -INFINITY;
      S.l[0] = S.l[1] = 0.f;
      {
        const bool hv = gid < G;
        const __nv_bfloat16* qrow = a.q + ((size_t)b * cv.Hq + kvh * G + (hv ? gid : 0)) * D + 32 * tq;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          S.bq[kk][0] = hv ? *(const uint32_t*)(qrow + 4 * kk) : 0u;
          S.bq[kk][1] = hv ? *(const uint32_t*)(qrow + 4 * kk + 2) : 0u;
        }
      }
      const size_t head = (size_t)b * Hkv + kvh;
      if (is_win) {
        const int Lq = sl[b];
        const int nsink = Lq < SINK ? Lq : SINK;
        const int recent = Lq > SINK ? Lq - SINK - hist_b : 0;
        const int h0 = hist_b % RECENT;
        // wch == 1: warps take the 5 chunks in turn; wch == 5: this item is
        // chunk wc and warp w takes its 16-token tile w
        const int ch_begin = wch == 1 ? warp : wc;
        const int ch_step = wch == 1 ? NW : 5;
        for (int ch = ch_begin; ch < 5; ch += ch_step) {
          uint64_t valid = 0;
          const __nv_bfloat16 *Kb, *Vb;
          if (ch == 0) {
            valid = nsink >= 64 ? ~0ull : ((1ull << nsink) - 1ull);
            Kb = cv.sink_k + head * SINK * D;
            Vb = cv.sink_v + head * SINK * D;
          } else {
            const int s0 = 64 * (ch - 1);
            // slots s0..s0+63 valid where (slot - h0) mod 256 < recent
#pragma unroll
            for (int half = 0; half < 2; ++half) {
              const int t = lane + 32 * half;
              const bool v = ((s0 + t - h0 + RECENT) % RECENT) < recent;
              const uint32_t bits = __ballot_sync(0xffffffffu, v);
              valid |= (uint64_t)bits << (32 * half);
            }
            Kb = cv.ring_k + (head * RECENT + s0) * D;
            Vb = cv.ring_v + (head * RECENT + s0) * D;
          }
          if (wch == 1) {
            if (valid) bf16_chunk_mma<BF16H>(S, Kb, Vb, valid, lane);
          } else if ((valid >> (16 * warp)) & 0xFFFFull) {
            bf16_span_mma<BF16H>(S, Kb, Vb, valid, lane, warp, 1);
          }
        }
      } else {
        const int nwp = (p1 - p0 - warp + NW - 1) / NW > 0 ? (p1 - p0 - warp + NW - 1) / NW : 0;
        PageIds P;
        page_ids_init(P, cv, b, p0 + warp, nwp, lane);
        for (int k = 0; k < nwp; ++k) {
          if (k > 0 && (k & 31) == 0) page_ids_advance(P, cv, b, p0 + warp, nwp, lane);
          const int p = p0 + warp + k * NW;
          const int pid = page_id_at(P, k);
          if (pid < 0 || pid >= cv.num_pages) {
            if (lane == 0) record_error(cv.err, pid < 0 ? OSCAR_ERR_NO_PAGE : OSCAR_ERR_RANGE);
            continue;
          }
          const int nv = (p == pages_b - 1) ? hist_b - p * PAGE : PAGE;
          const uint64_t valid = nv >= 64 ? ~0ull : ((1ull << nv) - 1ull);
          const __nv_bfloat16* Kb =
              (const __nv_bfloat16*)(cv.pool + (size_t)pid * cv.page_bytes + (size_t)kvh * BF16_HEAD_BYTES);
          bf16_chunk_mma<BF16H>(S, Kb, Kb + PAGE * D, valid, lane);
        }
      }
#pragma unroll
      for (int hc = 0; hc < 2; ++hc) {
        S.l[hc] += __shfl_xor_sync(0xffffffffu, S.l[hc], 4);
        S.l[hc] += __shfl_xor_sync(0xffffffffu, S.l[hc], 8);
        S.l[hc] += __shfl_xor_sync(0xffffffffu, S.l[hc], 16);
      }
      __syncthreads();  // everyone is done with the stage area
#pragma unroll
      for (int hc = 0; hc < 2; ++hc) {
        const int n = 2 * tq + hc;
        if (n < G) {
          if (gid == 0) {
            wm[warp * MAX_G + n] = S.m[hc];
            wl[warp * MAX_G + n] = S.l[hc];
          }
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            wo[(warp * MAX_G + n) * D + 16 * gid + 2 * j] = S.oacc[j][hc];
            wo[(warp * MAX_G + n) * D + 16 * gid + 2 * j + 1] = S.oacc[j][hc + 2];
          }
        }
      }
    } else if constexpr (!BF16H) {
      // ------------------------------------------------------ INT2 history
      const int nw_pages = (p1 - p0 - warp + NW - 1) / NW > 0 ? (p1 - p0 - warp + NW - 1) / NW : 0;
      uint8_t* my_stage = smem + L.off_stage + (size_t)warp * DEPTH * L.stage_bytes;
      uint64_t* my_bar = mbar + warp * DEPTH;
      PageIds P;
      page_ids_init(P, cv, b, p0 + warp, nw_pages, lane);
      auto issue = [&](int k, int pid) {  // lane 0 only: k-th page of this warp
        const int st = (int)((seq + k) % DEPTH);
        if (pid >= 0 && pid < cv.num_pages) {
          mbar_expect_tx(&my_bar[st], (uint32_t)cv.head_bytes);
          bulk_g2s_hint(my_stage + (size_t)st * L.stage_bytes,
                        cv.pool + (size_t)pid * cv.page_bytes + (size_t)kvh * cv.head_bytes,
                        (uint32_t)cv.head_bytes, &my_bar[st], l2_evict_first_policy());
        } else {
          record_error(cv.err, pid < 0 ? OSCAR_ERR_NO_PAGE : OSCAR_ERR_RANGE);
          mbar_expect_tx(&my_bar[st], 0u);
        }
      };
      __syncthreads();  // the previous item's results in the stage area are consumed
      if (lane == 0) fence_proxy_async();
      // the tensor-core paths issue their first page pair now (overlapping
      // prep_kernel) and the rest once the packed query is in shared memory,
      // so that its load does not queue behind a full wave of page copies
      constexpr int EARLY = (IMPL == 1) ? DEPTH : 2;
      // in a decode step the page that receives the demoted token is written
      // by the step kernel: it is copied only after the wait
      const int late_page = (a.step_pred && !waited && hl[b] > a.pred[2 * a.B + b]) ? a.pred[2 * a.B + b] / PAGE : -1;
      int deferred = -1;
      for (int k = 0; k < EARLY && k < nw_pages; ++k) {
        const int pid = page_id_at(P, k);
        if (p0 + warp + k * NW == late_page) {
          deferred = k;
          continue;
        }
        if (lane == 0) issue(k, pid);
      }
      if (!waited) {
        wait_prev();  // q' (prep or step kernel) is ready from here on
        waited = true;
      }
      if (deferred >= 0) {
        const int pid = page_id_at(P, deferred);
        if (lane == 0) issue(deferred, pid);
      }
      bool timed_out = false;
      int k_fail = 0;
      if constexpr (IMPL == 0 || IMPL == 3 || IMPL == 4) {
        // IMPL 3: pages in pairs, two streams per tile (G <= 4), with the codes
        // as fp16 subnormals; IMPL 0: one page at a time; IMPL 4: one page at
        // a time with the layer's Lloyd-Max codebook
        constexpr bool PAIR = (IMPL == 3);
        constexpr bool CB = (IMPL == 4);
        constexpr int QREC = CB ? QPACK_CB_BYTES : QPACK_BYTES;
        // the kv head's G packed query records, copied to shared memory by warp
        // 0 with coalesced 16-byte loads (every warp of every CTA reads them;
        // scattered per-lane loads pile the whole grid onto a few L2 lines,
        // and a bulk copy would queue behind this CTA's page copies)
        if (warp == 0) {
          const uint4* src = (const uint4*)(a.qpack + ((size_t)b * cv.Hq + kvh * G) * QREC);
          for (int e = lane; e < G * QREC / 16; e += 32) ((uint4*)qpk)[e] = __ldcg(src + e);
        }
        for (int k = EARLY; k < DEPTH && k < nw_pages; ++k) {
          const int pid = page_id_at(P, k);
          if (lane == 0) issue(k, pid);
        }
        __syncthreads();
        Int2State<NG> S;
        CbExtra X;
#pragma unroll
        for (int j = 0; j < 8; ++j) S.oacc[j][0] = S.oacc[j][1] = S.oacc[j][2] = S.oacc[j][3] = 0.f;
        {
          constexpr int O_ALPHA = CB ? QPACK_CB_ALPHA : QPACK_ALPHA;
          constexpr int O_PSUM = CB ? QPACK_CB_PSUM : QPACK_PSUM;
          float kc0 = 0.f;  // codebook: c0_K, the level of code 0
          if constexpr (CB) {
            const float* ck = a.rot.cb + (size_t)kvh * CB_WORDS;
            const float* cvr = a.rot.cb + (size_t)(Hkv + kvh) * CB_WORDS;
            kc0 = __ldg(ck + CB_C0);
            X.va = __ldg(cvr + CB_ALPHA);
            X.vb = __ldg(cvr + CB_BETA_HALF);
            X.vc0 = __ldg(cvr + CB_C0);
          }
          // B column gid carries head gid (PAIR: head gid & 3 in both halves)
          const int qh = PAIR ? (gid & 3) : gid;
          const bool qv = qh < G;
          const __half* qbh = (const __half*)(qpk + (qv ? qh : 0) * QREC);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            S.bq[kk][0] = qv ? *(const unsigned int*)(qbh + 16 * kk + 2 * tq) : 0u;
            S.bq[kk][1] = qv ? *(const unsigned int*)(qbh + 16 * kk + 8 + 2 * tq) : 0u;
            if constexpr (CB) {
              const __half* q2 = qbh + QPACK_CB_QB / 2;
              X.bq2[kk][0] = qv ? *(const unsigned int*)(q2 + 16 * kk + 2 * tq) : 0u;
              X.bq2[kk][1] = qv ? *(const unsigned int*)(q2 + 16 * kk + 8 + 2 * tq) : 0u;
            }
          }
#pragma unroll
          for (int hc = 0; hc < 2; ++hc) {
            const int n = PAIR ? ((2 * tq + hc) & 3) : 2 * tq + hc;
            const bool hv = n < G;
            const uint8_t* r = qpk + (hv ? n : 0) * QREC;
            S.m[hc] = PAIR ? -1e30f : -INFINITY;
            S.l[hc] = 0.f;
            const float al = hv ? *(const float*)(r + O_ALPHA) : 0.f;
            S.ka[hc] = al * 16777216.f;  // subnormal codes carry 2^-24
#pragma unroll
            for (int gr = 0; gr < NG; ++gr) {
              float ps = 0.f;
#pragma unroll
              for (int k = gr * (4 / NG); k < (gr + 1) * (4 / NG); ++k)
                ps += hv ? ((const float*)(r + O_PSUM))[k] : 0.f;
              S.zs[hc][gr] = 0.f;
              S.kb[hc][gr] = CB ? kc0 * ps * (LOG2E * INV_SQRT_D) : 0.f;
              S.kg[hc][gr] = ps * LOG2E * INV_SQRT_D;
            }
          }
        }
        if constexpr (PAIR) {
          const uint32_t mA = gid < 4 ? 0xffffffffu : 0u;  // B columns 0..3: page A
          for (int k = 0; k < nw_pages; k += 2) {
            const bool hasB = k + 1 < nw_pages;
            const int sa = (int)((seq + k) % DEPTH), sb = (int)((seq + k + 1) % DEPTH);
            bool ok = mbar_wait2(&my_bar[sa], ((seq + k) / DEPTH) & 1u, &my_bar[hasB ? sb : sa],
                                 (hasB ? (seq + k + 1) / DEPTH : (seq + k) / DEPTH) & 1u, a.wait_polls);
            if (!__all_sync(0xffffffffu, ok)) {
              timed_out = true;
              k_fail = k;
              break;
            }
            if (k > 0 && (k & 31) == 0) page_ids_advance(P, cv, b, p0 + warp, nw_pages, lane);
            const int pa = p0 + warp + k * NW, pb = pa + NW;
            const int pida = page_id_at(P, k);
            const int pidb = page_id_at(P, hasB ? k + 1 : k);
            const bool oka = pida >= 0 && pida < cv.num_pages;
            const bool okb = hasB && pidb >= 0 && pidb < cv.num_pages;
            const int nva = oka ? ((pa == pages_b - 1) ? hist_b - pa * PAGE : PAGE) : 0;
            const int nvb = okb ? ((pb == pages_b - 1) ? hist_b - pb * PAGE : PAGE) : 0;
            const uint8_t* sta = my_stage + (size_t)sa * L.stage_bytes;
            const uint8_t* stb = hasB ? my_stage + (size_t)sb * L.stage_bytes : sta;
            // one (masked) variant for full and partial pages keeps the
            // unrolled loop body small enough for the instruction cache
            if (nva > 0 || nvb > 0) int2_pair_mma<NG, false>(S, sta, nva, stb, nvb, hasB, lane, mA);
            __syncwarp();
#pragma unroll
            for (int u = 0; u < 2; ++u) {
              if (k + u + DEPTH < nw_pages) {
                // the stage's generic-proxy reads have completed (their values
                // were consumed before __syncwarp): no proxy fence is needed
                const int pid_next = page_id_at(P, k + u + DEPTH);
                if (lane == 0) issue(k + u + DEPTH, pid_next);
              }
            }
          }
        } else {
          for (int k = 0; k < nw_pages; ++k) {
            const int st = (int)((seq + k) % DEPTH);
            const uint32_t ph = ((seq + k) / DEPTH) & 1u;
            if (!__all_sync(0xffffffffu, mbar_wait(&my_bar[st], ph, a.wait_polls))) {
              timed_out = true;
              k_fail = k;
              break;
            }
            if (k > 0 && (k & 31) == 0) page_ids_advance(P, cv, b, p0 + warp, nw_pages, lane);
            const int p = p0 + warp + k * NW;
            const int pid = page_id_at(P, k);
            if (pid >= 0 && pid < cv.num_pages) {
              const int nv = (p == pages_b - 1) ? hist_b - p * PAGE : PAGE;
              if constexpr (CB) {
                if (nv == PAGE)
                  int2_page_mma_cb<NG, true>(S, X, my_stage + (size_t)st * L.stage_bytes, nv, lane);
                else
                  int2_page_mma_cb<NG, false>(S, X, my_stage + (size_t)st * L.stage_bytes, nv, lane);
              } else if (nv == PAGE) {
                int2_page_mma<NG, true>(S, my_stage + (size_t)st * L.stage_bytes, nv, lane);
              } else {
                int2_page_mma<NG, false>(S, my_stage + (size_t)st * L.stage_bytes, nv, lane);
              }
            }
            __syncwarp();
            if (k + DEPTH < nw_pages) {
              const int pid_next = page_id_at(P, k + DEPTH);
              if (lane == 0) issue(k + DEPTH, pid_next);  // reads of the stage are complete
            }
          }
        }
#pragma unroll
        for (int hc = 0; hc < 2; ++hc) {
#pragma unroll
          for (int o = 4; o < 32; o <<= 1) {
            S.l[hc] += __shfl_xor_sync(0xffffffffu, S.l[hc], o);
#pragma unroll
            for (int gr = 0; gr < NG; ++gr) {
              S.zs[hc][gr] += __shfl_xor_sync(0xffffffffu, S.zs[hc][gr], o);
            }
          }
        }
        if constexpr (PAIR) merge_pair_streams<NG>(S);
        if (timed_out) {
          if (lane == 0) {
            record_error(cv.err, OSCAR_ERR_TIMEOUT);
            misc[1] = 1;
          }
          const int issued = (k_fail + DEPTH) < nw_pages ? k_fail + DEPTH : nw_pages;
          for (int kk = k_fail; kk < issued; ++kk)
            mbar_wait(&my_bar[(seq + kk) % DEPTH], ((seq + kk) / DEPTH) & 1u);
        }
        __syncthreads();  // all warps are past their stages: results may alias them
#pragma unroll
        for (int hc = 0; hc < 2; ++hc) {
          const int n = 2 * tq + hc;
          if (n < G) {
            if (gid == 0) {
              wm[warp * MAX_G + n] = S.m[hc];
              wl[warp * MAX_G + n] = S.l[hc];
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const int gr = j / (8 / NG);
              // subnormal codes: o' = 2^16 O + sum p z
              const float z = S.zs[hc][gr];
              wo[(warp * MAX_G + n) * D + 16 * j + gid] = fmaf(S.oacc[j][hc], 65536.f, z);
              wo[(warp * MAX_G + n) * D + 16 * j + 8 + gid] = fmaf(S.oacc[j][hc + 2], 65536.f, z);
            }
          }
        }
      } else {
        // CUDA-core path: q' in K storage order and the z weights, in smem
        float* kgm = qf + MAX_G * D;
        for (int e = threadIdx.x; e < G * D; e += NW * 32) {
          const int n = e / D, c = e % D;
          qf[n * D + k_word(c) * 16 + k_bit(c) / 2] =
              __ldcg(a.qrot + ((size_t)b * cv.Hq + kvh * G + n) * D + c);
        }
        for (int e = threadIdx.x; e < G * 4; e += NW * 32) {
          const int n = e / 4, gr = e % 4;
          const float* ps = (const float*)(a.qpack + ((size_t)b * cv.Hq + kvh * G + n) * QPACK_BYTES + QPACK_PSUM);
          float sum = 0.f;
          if (gr < NG)
            for (int k = gr * (4 / NG); k < (gr + 1) * (4 / NG); ++k) sum += __ldcg(ps + k);
          kgm[e] = sum * LOG2E * INV_SQRT_D;
        }
        __syncthreads();
        CoreState S;
        for (int n = 0; n < MAX_G; ++n) {
          S.m[n] = -INFINITY;
          S.l[n] = 0.f;
#pragma unroll
          for (int c = 0; c < 4; ++c) S.o[n][c] = 0.f;
        }
        float* ps = vsw + warp * (MAX_G * PAGE + 2 * 4 * PAGE);
        float* vs = ps + MAX_G * PAGE;
        for (int k = 0; k < nw_pages; ++k) {
          const int st = (int)((seq + k) % DEPTH);
          const uint32_t ph = ((seq + k) / DEPTH) & 1u;
          if (!__all_sync(0xffffffffu, mbar_wait(&my_bar[st], ph, a.wait_polls))) {
            timed_out = true;
            k_fail = k;
            break;
          }
          if (k > 0 && (k & 31) == 0) page_ids_advance(P, cv, b, p0 + warp, nw_pages, lane);
          const int p = p0 + warp + k * NW;
          const int pid = page_id_at(P, k);
          if (pid >= 0 && pid < cv.num_pages) {
            const int nv = (p == pages_b - 1) ? hist_b - p * PAGE : PAGE;
            int2_page_core<NG>(S, my_stage + (size_t)st * L.stage_bytes, nv, lane, G, qf, kgm, ps, vs);
          }
          __syncwarp();
          if (k + DEPTH < nw_pages) {
            const int pid_next = page_id_at(P, k + DEPTH);
            if (lane == 0) issue(k + DEPTH, pid_next);  // reads of the stage are complete
          }
        }
        if (timed_out) {
          if (lane == 0) {
            record_error(cv.err, OSCAR_ERR_TIMEOUT);
            misc[1] = 1;
          }
          const int issued = (k_fail + DEPTH) < nw_pages ? k_fail + DEPTH : nw_pages;
          for (int kk = k_fail; kk < issued; ++kk)
            mbar_wait(&my_bar[(seq + kk) % DEPTH], ((seq + kk) / DEPTH) & 1u);
        }
        __syncthreads();
        for (int n = 0; n < G; ++n) {
          if (lane == 0) {
            wm[warp * MAX_G + n] = S.m[n];
            wl[warp * MAX_G + n] = S.l[n];
          }
#pragma unroll
          for (int c = 0; c < 4; ++c) wo[(warp * MAX_G + n) * D + 4 * lane + c] = S.o[n][c];
        }
      }
      seq += (uint32_t)nw_pages;
    }
    __syncthreads();
    cta_combine_write(a, wm, wl, wo, slot);
    if (!waited) {
      wait_prev();
      waited = true;
    }
    if (misc[1]) break;
    __syncthreads();  // every thread has read the item before thread 0 moves on
    if (threadIdx.x == 0) {
      if (bal) cursor_next(*cur, a.B, Hkv, (long long*)pre, hl, sl);
      else misc[0] = (int)gridDim.x + atomicAdd(a.counter, 1);
    }
    __syncthreads();
    it = misc[0];
  }
  if (!waited) wait_prev();
}

// Raise decode_kernel<NG, IMPL>'s dynamic shared-memory limit to `bytes` if it
// is lower (never lowered: launches and occupancy queries of other sizes
// share it).
template <int NG, int IMPL>
cudaError_t ensure_decode_smem(int bytes) {
  static int limit[MAX_DEVICES];
  return raise_smem_limit(decode_kernel<NG, IMPL>, limit, bytes);
}

template <int NG, int IMPL>
cudaError_t launch_decode_t(const DecodeArgs& a, int grid, cudaStream_t st) {
  const SmemLayout L = smem_layout(a.cv.head_bytes, a.B, IMPL, a.cv.G);
  if ((L.off_mbar % 8) || (L.off_stage % 128) || (L.off_pre % 16) || (L.off_qpk % 16)) return cudaErrorInvalidValue;
  const cudaError_t e = ensure_decode_smem<NG, IMPL>(L.total);
  if (e != cudaSuccess) return e;
  return launch_pdl(decode_kernel<NG, IMPL>, dim3(grid), dim3(NW * 32), L.total, st, a);
}

cudaError_t launch_merge(const DecodeArgs& a, cudaStream_t st) {
  const MergeLayout ML = merge_layout(a.B);
  if ((ML.off_mbar % 8) || (ML.off_y % 16) || (ML.off_to % 16) || (ML.off_wo % 16)) return cudaErrorInvalidValue;
  if (a.merge_hpc < 1 || a.cv.G % a.merge_hpc) return cudaErrorInvalidValue;
  static int limit[MAX_DEVICES];
  const cudaError_t e = raise_smem_limit(merge_kernel, limit, ML.total);
  if (e != cudaSuccess) return e;
  return launch_pdl(merge_kernel, dim3(a.B * a.cv.Hkv * (a.cv.G / a.merge_hpc)), dim3(MW * 32), ML.total, st, a);
}

}  // namespace

ScratchLayout scratch_layout(int B, int Hq, int Hkv, int G, int max_target_items) {
  auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
  ScratchLayout s;
  s.off_counter = 0;
  s.off_pred = 256;
  s.off_qrot = s.off_pred + up((size_t)3 * B * 4);
  s.off_qpack = s.off_qrot + up((size_t)B * Hq * D * 4);
  s.off_part = s.off_qpack + up((size_t)B * Hq * QPACK_CB_BYTES);  // room for codebook records
  const size_t slots = (size_t)max_target_items + 2 * (size_t)B * Hkv;
  s.total = s.off_part + slots * G * PART_STRIDE * 4;
  return s;
}

size_t decode_scratch_bytes(int B, int Hq, int Hkv, int G, int max_target_items) {
  return scratch_layout(B, Hq, Hkv, G, max_target_items).total;
}

// Resident decode CTAs per SM for this launch's kernel and shared memory
// (cached per kernel variant and shared-memory size).
template <int NG, int IMPL>
int occupancy_t(const DecodeArgs& a) {
  static int cached_smem[MAX_DEVICES], cached_occ[MAX_DEVICES];
  const SmemLayout L = smem_layout(a.cv.head_bytes, a.B, IMPL, a.cv.G);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) {
    (void)cudaGetLastError();
    return 0;
  }
  if (cached_smem[dev] == L.total) return cached_occ[dev];
  if (ensure_decode_smem<NG, IMPL>(L.total) != cudaSuccess) {
    (void)cudaGetLastError();
    return 0;
  }
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_kernel<NG, IMPL>, NW * 32, L.total) !=
      cudaSuccess) {
    (void)cudaGetLastError();
    return 0;
  }
  cached_occ[dev] = n;
  cached_smem[dev] = L.total;
  return n;
}

int decode_ctas_per_sm(const DecodeArgs& a) {
  const int NG = a.cv.NG;
  if (a.bf16_history) return occupancy_t<1, 2>(a);
  if (a.impl == 5) return 1;  // the tensor-memory kernel holds all of an SM's tensor memory
  if (a.impl == 1) return NG == 1 ? occupancy_t<1, 1>(a) : NG == 2 ? occupancy_t<2, 1>(a) : occupancy_t<4, 1>(a);
  if (a.impl == 3) return NG == 1 ? occupancy_t<1, 3>(a) : NG == 2 ? occupancy_t<2, 3>(a) : occupancy_t<4, 3>(a);
  if (a.impl == 4) return NG == 1 ? occupancy_t<1, 4>(a) : NG == 2 ? occupancy_t<2, 4>(a) : occupancy_t<4, 4>(a);
  return NG == 1 ? occupancy_t<1, 0>(a) : NG == 2 ? occupancy_t<2, 0>(a) : occupancy_t<4, 0>(a);
}

cudaError_t launch_decode_after_prep(const DecodeArgs& a, int grid, cudaStream_t st, Profiler* prof) {
  const CacheView& cv = a.cv;
  cudaError_t e;
  prof_begin(prof, OSCAR_KERNEL_DECODE_MAIN, st);
  if (a.impl == 5 && !a.bf16_history) {
    e = launch_decode_tc(a, st);
  } else if (a.bf16_history) {
    e = launch_decode_t<1, 2>(a, grid, st);
  } else if (a.impl == 1) {
    if (cv.NG == 1) e = launch_decode_t<1, 1>(a, grid, st);
    else if (cv.NG == 2) e = launch_decode_t<2, 1>(a, grid, st);
    else e = launch_decode_t<4, 1>(a, grid, st);
  } else if (a.impl == 3) {
    if (cv.NG == 1) e = launch_decode_t<1, 3>(a, grid, st);
    else if (cv.NG == 2) e = launch_decode_t<2, 3>(a, grid, st);
    else e = launch_decode_t<4, 3>(a, grid, st);
  } else if (a.impl == 4) {
    if (cv.NG == 1) e = launch_decode_t<1, 4>(a, grid, st);
    else if (cv.NG == 2) e = launch_decode_t<2, 4>(a, grid, st);
    else e = launch_decode_t<4, 4>(a, grid, st);
  } else {
    if (cv.NG == 1) e = launch_decode_t<1, 0>(a, grid, st);
    else if (cv.NG == 2) e = launch_decode_t<2, 0>(a, grid, st);
    else e = launch_decode_t<4, 0>(a, grid, st);
  }
  prof_end(prof, OSCAR_KERNEL_DECODE_MAIN, st);
  if (e != cudaSuccess) return e;
  prof_begin(prof, OSCAR_KERNEL_DECODE_MERGE, st);
  e = launch_merge(a, st);
  prof_end(prof, OSCAR_KERNEL_DECODE_MERGE, st);
  return e;
}

cudaError_t launch_decode(const DecodeArgs& a, int grid, cudaStream_t st, Profiler* prof) {
  prof_begin(prof, OSCAR_KERNEL_DECODE_PREP, st);
  const cudaError_t e = launch_pdl(prep_kernel, dim3(a.B * a.cv.Hkv, 4), dim3(128), 0, st, a);
  prof_end(prof, OSCAR_KERNEL_DECODE_PREP, st);
  if (e != cudaSuccess) return e;
  return launch_decode_after_prep(a, grid, st, prof);
}

}  // namespace oscar
