// Chunked prefill over the three-region cache (sm_103a): the T new tokens of
// each request attend to its BF16 sink and recent window, to its INT2 history
// in the rotated basis, and causally to one another; the chunk itself is not
// stored.  This is the prefix-hit extension of the cache layout in [News,
// "服务系统：混合精度缓存布局"] with the attention of [Blog, pipeline figure
// paragraph]: logits q'·k'/sqrt(d) with q' = q·R_K against the dequantised
// history, the history output un-rotated by R_V^T, one softmax over all
// regions.
//
// Three kernels on one stream, each a programmatic dependent of the last:
//  prefill_prep_kernel   per query row (token t, head h of a kv head; row
//                        r = t·G + h): q·R_K and q, both scaled by 2^-sigma
//                        into fp16, and the logit factor 2^sigma·log2(e)/sqrt(d)
//  prefill_attn_kernel   per (request, kv head, 128-row tile): NS CTAs over
//                        slices of the history pages and one over the window
//                        (sink, ring, chunk); 8 warps x 16 rows, flash-attention
//                        style on tensor cores.  INT2 pages arrive by bulk
//                        copy and are dequantised (s·code + z, fp16) once per
//                        CTA into shared tiles that all 8 warps read, so the
//                        unpacking is spread over 128 query rows.
//  prefill_merge_kernel  per 8 rows: combines the history slices, un-rotates
//                        them by R_V^T and merges the window partial.
#include "oscar_internal.cuh"

namespace oscar {
namespace {

constexpr int PF_WARPS = 8;
constexpr int PF_THREADS = 32 * PF_WARPS;
constexpr int PF_DEPTH = 4;               // INT2 pages in flight per CTA
constexpr int TILE_BYTES = PAGE * D * 2;  // one fp16 tile: K [64][128] or V^T [128][64]
constexpr int RAW_SLOT = 6144;            // largest INT2 head block (g = 32)
// dynamic shared memory of prefill_attn_kernel
constexpr int OFF_TILES = 0;  // [2 buffers][K tile, V^T tile], 16-byte chunks XOR-swizzled by row
constexpr int OFF_RAW = 4 * TILE_BYTES;
constexpr int OFF_BAR = OFF_RAW + PF_DEPTH * RAW_SLOT;
constexpr int OFF_INFO = OFF_BAR + PF_DEPTH * 8;  // u64 mask[2], int causal[2], int bad[PF_DEPTH]
constexpr int PF_SMEM = OFF_INFO + 64;
static_assert(RAW_SLOT >= int2_head_bytes(32), "raw slot holds a g32 head block");

__device__ __forceinline__ uint32_t hfma2u(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("fma.rn.f16x2 %0, %1, %2, %3;\n" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

__device__ __forceinline__ uint32_t f2_to_h2(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;\n" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// The code pair at bit pair I of each 16-bit half of w as exact f16x2 values
// 0..3: code_pair gives 1024 + code·2^E, and (h - 1024)·2^-E is exact.
template <int I>
__device__ __forceinline__ uint32_t codes_f16x2(uint32_t w) {
  constexpr int E = code_exp<I>();
  constexpr uint32_t SC = E == 4 ? 0x2C002C00u : E == 6 ? 0x24002400u : 0x1C001C00u;   // 2^-E
  constexpr uint32_t OF = E == 4 ? 0xD400D400u : E == 6 ? 0xCC00CC00u : 0xC400C400u;   // -1024·2^-E
  return hfma2u(code_pair<I>(w), SC, OF);
}

// Lloyd-Max codebook of one side (keys or values) of the item's kv head as
// f16x2 constants: level(code) = c0 + alpha*bit0 + beta_half*(2*bit1).
struct CbLevels {
  uint32_t c0, al, bh;
};

__device__ __forceinline__ CbLevels cb_levels(const float* rec) {
  CbLevels L;
  const __half2 c0 = __float2half2_rn(__ldg(rec + CB_C0));
  const __half2 al = __float2half2_rn(__ldg(rec + CB_ALPHA));
  const __half2 bh = __float2half2_rn(__ldg(rec + CB_BETA_HALF));
  L.c0 = *(const uint32_t*)&c0;
  L.al = *(const uint32_t*)&al;
  L.bh = *(const uint32_t*)&bh;
  return L;
}

// The levels of code_pair<I>'s two codes: each bit plane gives its bit
// exactly (0 or 1, and 0 or 2 for the high bit), then two fp16 FMAs.
template <int I>
__device__ __forceinline__ uint32_t levels_f16x2(uint32_t w, const CbLevels& L) {
  constexpr int E = code_exp<I>();
  constexpr uint32_t SC = E == 4 ? 0x2C002C00u : E == 6 ? 0x24002400u : 0x1C001C00u;   // 2^-E
  constexpr uint32_t OF = E == 4 ? 0xD400D400u : E == 6 ? 0xCC00CC00u : 0xC400C400u;   // -1024·2^-E
  const uint32_t b0 = hfma2u(code_plane<I, 0>(w), SC, OF);
  const uint32_t b1x2 = hfma2u(code_plane<I, 1>(w), SC, OF);
  return hfma2u(b1x2, L.bh, hfma2u(b0, L.al, L.c0));
}

// ------------------------------------------------------------ tile filling
// K tile: row = token (256 B), 16-byte chunk j of row t stored at j ^ (t & 7).
// V^T tile: row = channel (128 B), chunk j of row c stored at j ^ (c & 7).
// Tokens outside the tile's valid set are written as zeros.

// Dequantise one INT2 head block (raw, in shared memory) into the K and V^T
// tiles: value = s·code + z with the group's fp16 scale and zero, rounded
// once to fp16 (CB: s·level(code) + z with the codebook's fp16 levels).
// nv = valid tokens (rows 0..nv-1).
template <int I, bool CB>
__device__ __forceinline__ void k_store(uint8_t* Kt, int tr, int A, int dq, uint32_t w, uint32_t s2,
                                        uint32_t z2, bool ok, const CbLevels& L) {
  const uint32_t c = CB ? levels_f16x2<I>(w, L) : codes_f16x2<I>(w);
  const uint32_t val = ok ? hfma2u(c, s2, z2) : 0u;
  *(uint32_t*)(Kt + tr * 256 + ((((8 * A + I) ^ (tr & 7))) << 4) + 4 * dq) = val;
}

template <int I, bool CB>
__device__ __forceinline__ void v_store(uint8_t* Vt, int ch, int T4, uint32_t w, const uint32_t* vsz,
                                        int NG, int grp, int nv, const CbLevels& L) {
  const int t = 8 * I + 2 * T4;  // token slot of the low half; t + 1 in the high half
  const uint32_t a = vsz[t * NG + grp], b = vsz[(t + 1) * NG + grp];
  const uint32_t c = CB ? levels_f16x2<I>(w, L) : codes_f16x2<I>(w);
  uint32_t val = hfma2u(c, prmt(a, b, 0x5410u), prmt(a, b, 0x7632u));
  if (t + 1 >= nv) val = t < nv ? (val & 0xFFFFu) : 0u;
  *(uint32_t*)(Vt + ch * 128 + (((I ^ (ch & 7))) << 4) + 4 * T4) = val;
}

template <bool CB>
__device__ __forceinline__ void fill_int2(uint8_t* smem, int buf, const uint8_t* raw, int g, int nv,
                                          const CbLevels& LK, const CbLevels& LV) {
  const int tid = threadIdx.x, NG = D / g;
  uint8_t* Kt = smem + OFF_TILES + buf * 2 * TILE_BYTES;
  uint8_t* Vt = Kt + TILE_BYTES;
  {  // K: token tr, words 2dq (A = 0) and 2dq + 1 (A = 1); channel c = 64A + 8I + 2dq + E
    const int tr = tid >> 2, dq = tid & 3;
    const uint2 cw = *(const uint2*)(raw + tr * 32 + 8 * dq);
    const uint32_t* ksz = (const uint32_t*)(raw + off_k_sz()) + tr * NG;
    const bool ok = tr < nv;
#pragma unroll
    for (int A = 0; A < 2; ++A) {
      const uint32_t w = A ? cw.y : cw.x;
      const uint32_t lo = ksz[(64 * A) / g], hi = ksz[(64 * A + 32) / g];  // groups of I < 4, I >= 4
      const uint32_t s0 = prmt(lo, lo, 0x1010u), z0 = prmt(lo, lo, 0x3232u);
      const uint32_t s1 = prmt(hi, hi, 0x1010u), z1 = prmt(hi, hi, 0x3232u);
      k_store<0, CB>(Kt, tr, A, dq, w, s0, z0, ok, LK);
      k_store<1, CB>(Kt, tr, A, dq, w, s0, z0, ok, LK);
      k_store<2, CB>(Kt, tr, A, dq, w, s0, z0, ok, LK);
      k_store<3, CB>(Kt, tr, A, dq, w, s0, z0, ok, LK);
      k_store<4, CB>(Kt, tr, A, dq, w, s1, z1, ok, LK);
      k_store<5, CB>(Kt, tr, A, dq, w, s1, z1, ok, LK);
      k_store<6, CB>(Kt, tr, A, dq, w, s1, z1, ok, LK);
      k_store<7, CB>(Kt, tr, A, dq, w, s1, z1, ok, LK);
    }
  }
  {  // V: channel ch, word T4 holds token slots 8I + 2T4 + E
    const int T4 = tid & 3;
    const uint32_t* vsz = (const uint32_t*)(raw + off_v_sz(g));
#pragma unroll
    for (int hc = 0; hc < 2; ++hc) {
      const int ch = (tid >> 2) + 64 * hc;
      const uint32_t w = *(const uint32_t*)(raw + 2048 + ch * 16 + 4 * T4);
      const int grp = ch / g;
      v_store<0, CB>(Vt, ch, T4, w, vsz, NG, grp, nv, LV);
      v_store<1, CB>(Vt, ch, T4, w, vsz, NG, grp, nv, LV);
      v_store<2, CB>(Vt, ch, T4, w, vsz, NG, grp, nv, LV);
      v_store<3, CB>(Vt, ch, T4, w, vsz, NG, grp, nv, LV);
      v_store<4, CB>(Vt, ch, T4, w, vsz, NG, grp, nv, LV);
      v_store<5, CB>(Vt, ch, T4, w, vsz, NG, grp, nv, LV);
      v_store<6, CB>(Vt, ch, T4, w, vsz, NG, grp, nv, LV);
      v_store<7, CB>(Vt, ch, T4, w, vsz, NG, grp, nv, LV);
    }
  }
}

__device__ __forceinline__ uint32_t bf2_to_h2(uint32_t x) {
  return f2_to_h2(__uint_as_float(x << 16), __uint_as_float(x & 0xFFFF0000u));
}

// Copy 64 BF16 tokens (row t at Kb + t·stride, Vb + t·stride) into the K and
// V^T tiles as fp16; rows whose bit in `valid` is clear become zeros.
__device__ __forceinline__ void fill_bf16(uint8_t* smem, int buf, const __nv_bfloat16* Kb,
                                          const __nv_bfloat16* Vb, size_t stride, uint64_t valid) {
  const int tid = threadIdx.x;
  uint8_t* Kt = smem + OFF_TILES + buf * 2 * TILE_BYTES;
  uint8_t* Vt = Kt + TILE_BYTES;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int u = tid + PF_THREADS * j, t = u >> 4, c16 = u & 15;
    uint4 x = make_uint4(0u, 0u, 0u, 0u);
    if ((valid >> t) & 1ull) x = *(const uint4*)(Kb + t * stride + 8 * c16);
    const uint4 y = make_uint4(bf2_to_h2(x.x), bf2_to_h2(x.y), bf2_to_h2(x.z), bf2_to_h2(x.w));
    *(uint4*)(Kt + t * 256 + ((c16 ^ (t & 7)) << 4)) = y;
  }
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const int u = tid + PF_THREADS * j, jp = u & 31, k8 = u >> 5;  // tokens 2jp, 2jp + 1; channels 8k8..
    uint4 x0 = make_uint4(0u, 0u, 0u, 0u), x1 = x0;
    if ((valid >> (2 * jp)) & 1ull) x0 = *(const uint4*)(Vb + (2 * jp) * stride + 8 * k8);
    if ((valid >> (2 * jp + 1)) & 1ull) x1 = *(const uint4*)(Vb + (2 * jp + 1) * stride + 8 * k8);
    const uint32_t a[4] = {x0.x, x0.y, x0.z, x0.w}, b[4] = {x1.x, x1.y, x1.z, x1.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t lo = i & 1 ? (a[i >> 1] & 0xFFFF0000u) : (a[i >> 1] << 16);
      const uint32_t hi = i & 1 ? (b[i >> 1] & 0xFFFF0000u) : (b[i >> 1] << 16);
      *(uint32_t*)(Vt + (8 * k8 + i) * 128 + ((((jp >> 2) ^ i)) << 4) + 4 * (jp & 3)) =
          f2_to_h2(__uint_as_float(lo), __uint_as_float(hi));
    }
  }
}

// ------------------------------------------------------------- attention
// Online-softmax state of one warp's 16 rows (rows gid and gid + 8 of the
// mma fragments), logits in log2 units.
struct RowState {
  float o[16][4];
  float m[2], l[2];
};

// One 64-token tile against the warp's 16 query rows: S = Q·K^T on tensor
// cores, scale and mask, online softmax, O += P·V.
__device__ __forceinline__ void tile_attend(RowState& st, const uint32_t (&qa)[8][4], const float (&al)[2],
                                            const int (&trow)[2], uint32_t kt_addr, uint32_t vt_addr,
                                            uint64_t mask, bool causal, int lane) {
  const int tig = lane & 3;
  float s[8][4];
#pragma unroll
  for (int n = 0; n < 8; ++n) s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
  // ldmatrix row addresses: matrix lane >> 3, row lane & 7
  const int mr = ((lane >> 4) << 3) + (lane & 7), mc = (lane >> 3) & 1;
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) {
#pragma unroll
    for (int np = 0; np < 4; ++np) {
      const int t = 16 * np + mr, c = 2 * ks + mc;
      uint32_t b0, b1, b2, b3;
      ldsm_x4(kt_addr + t * 256 + ((c ^ (t & 7)) << 4), b0, b1, b2, b3);
      mma_f16(s[2 * np], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b0, b1);
      mma_f16(s[2 * np + 1], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b2, b3);
    }
  }
  float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
  for (int n = 0; n < 8; ++n) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int col = 8 * n + 2 * tig + (e & 1), h = e >> 1;
      const bool ok = ((mask >> col) & 1ull) && !(causal && col > trow[h]);
      s[n][e] = ok ? s[n][e] * al[h] : -INFINITY;
      mx[h] = fmaxf(mx[h], s[n][e]);
    }
  }
  float sc[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 1));
    mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 2));
    const float mn = fmaxf(st.m[h], mx[h]);
    sc[h] = ex2(st.m[h] - mn);
    st.m[h] = mn;
    st.l[h] *= sc[h];
  }
#pragma unroll
  for (int n = 0; n < 16; ++n) {
    st.o[n][0] *= sc[0];
    st.o[n][1] *= sc[0];
    st.o[n][2] *= sc[1];
    st.o[n][3] *= sc[1];
  }
  uint32_t pa[4][4];
#pragma unroll
  for (int n = 0; n < 8; ++n) {
    const float p0 = ex2(s[n][0] - st.m[0]), p1 = ex2(s[n][1] - st.m[0]);
    const float p2 = ex2(s[n][2] - st.m[1]), p3 = ex2(s[n][3] - st.m[1]);
    st.l[0] += p0 + p1;
    st.l[1] += p2 + p3;
    pa[n >> 1][(n & 1) * 2 + 0] = f2_to_h2(p0, p1);
    pa[n >> 1][(n & 1) * 2 + 1] = f2_to_h2(p2, p3);
  }
#pragma unroll
  for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
    for (int np = 0; np < 8; ++np) {
      const int ch = 16 * np + mr, c = 2 * kk + mc;
      uint32_t b0, b1, b2, b3;
      ldsm_x4(vt_addr + ch * 128 + ((c ^ (ch & 7)) << 4), b0, b1, b2, b3);
      mma_f16(st.o[2 * np], pa[kk][0], pa[kk][1], pa[kk][2], pa[kk][3], b0, b1);
      mma_f16(st.o[2 * np + 1], pa[kk][0], pa[kk][1], pa[kk][2], pa[kk][3], b2, b3);
    }
  }
}

__device__ __forceinline__ uint64_t low_mask(int n) {
  return n >= 64 ? ~0ull : n <= 0 ? 0ull : ((1ull << n) - 1ull);
}

// --------------------------------------------------------------- kernels
constexpr int PREP_ROWS = 16;  // query rows per prep CTA
constexpr int PREP_SMEM = (D * D + PREP_ROWS * D + PREP_ROWS) * 4;

// 16 query rows of one kv head by 256 threads: thread (c, h) forms channel c
// of rows 8h .. 8h + 7 from the R_K staged in shared memory.
__global__ void __launch_bounds__(256) prefill_prep_kernel(PrefillArgs a) {
  extern __shared__ __align__(16) float psm[];
  float* Rs = psm;              // [128][128] R_K
  float* xs = Rs + D * D;       // [16][128] q rows
  float* nrm = xs + PREP_ROWS * D;
  const CacheView& cv = a.cv;
  const int bk = blockIdx.x, b = bk / cv.Hkv, kvh = bk % cv.Hkv, G = cv.G;
  const int R = a.T * G, RP = a.RT * PF_ROWS, r0 = PREP_ROWS * blockIdx.y;
  const int tid = threadIdx.x, c = tid & 127, h = tid >> 7, w = tid >> 5, lane = tid & 31;
  const int lgG = __ffs(G) - 1;  // G is a power of two
  {  // the rotation table is written synchronously by oscar_set_rotation: load it before the wait
    const float4* Rg = (const float4*)(a.rot.R_K + (size_t)kvh * D * D);
    float4 rv[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) rv[j] = __ldg(Rg + tid + 256 * j);
#pragma unroll
    for (int j = 0; j < 16; ++j) ((float4*)Rs)[tid + 256 * j] = rv[j];
  }
  pdl_wait();
  pdl_launch_dependents();
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int r = r0 + 8 * h + j;
    xs[(8 * h + j) * D + c] =
        r < R ? __bfloat162float(a.q[(((size_t)b * a.T + (r >> lgG)) * cv.Hq + kvh * G + (r & (G - 1))) * D + c])
              : 0.f;
  }
  __syncthreads();
#pragma unroll
  for (int jj = 0; jj < 2; ++jj) {
    const int j = 2 * w + jj;
    float sq = 0.f;
#pragma unroll
    for (int k = 0; k < 4; ++k) sq = fmaf(xs[j * D + lane + 32 * k], xs[j * D + lane + 32 * k], sq);
#pragma unroll
    for (int o = 16; o; o >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, o);
    if (lane == 0) nrm[j] = sqrtf(sq);
  }
  __syncthreads();
  float acc[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) acc[j] = 0.f;
  const float* xh = xs + 8 * h * D;
#pragma unroll 2
  for (int k = 0; k < D; k += 4) {
    const float r0 = Rs[k * D + c], r1 = Rs[(k + 1) * D + c], r2 = Rs[(k + 2) * D + c], r3 = Rs[(k + 3) * D + c];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float4 x = *(const float4*)(xh + j * D + k);  // same address across the warp: one broadcast
      acc[j] = fmaf(x.x, r0, fmaf(x.y, r1, fmaf(x.z, r2, fmaf(x.w, r3, acc[j]))));
    }
  }
  const size_t vstride = (size_t)a.B * cv.Hkv * RP * D;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int r = r0 + 8 * h + j;
    const float nj = nrm[8 * h + j];
    // |q'_c| and |q_c| are both at most |q| (R_K is orthogonal): 2^-sigma
    // brings them below 2^14 in fp16 (exact power-of-two scalings)
    const int ex = ((__float_as_int(nj) >> 23) & 0xFF) - 126;  // nj = m·2^ex, m in [0.5, 1)
    const int sig = nj > 0.f ? min(max(ex - 14, -120), 120) : 0;  // 2^±sig stay normal floats
    const float down = __int_as_float((127 - sig) << 23), up = __int_as_float((127 + sig) << 23);
    const size_t e = ((size_t)bk * RP + r) * D + c;
    a.qh[e] = __float2half_rn(acc[j] * down);
    a.qh[vstride + e] = __float2half_rn(xh[j * D + c] * down);
    if (c == 0) a.alpha[(size_t)bk * RP + r] = up * LOG2E * INV_SQRT_D;
  }
}

__global__ void __launch_bounds__(PF_THREADS, 1) prefill_attn_kernel(PrefillArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  const CacheView& cv = a.cv;
  const int Hkv = cv.Hkv, G = cv.G;
  const int tile = blockIdx.x, bk = tile / a.RT, rt = tile % a.RT;
  const int b = bk / Hkv, kvh = bk % Hkv;
  const int split = blockIdx.y;
  const bool win = split == a.NS;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, gid = lane >> 2, tig = lane & 3;
  const int R = a.T * G, RP = a.RT * PF_ROWS;
  uint64_t* bars = (uint64_t*)(smem + OFF_BAR);
  uint64_t* tmask = (uint64_t*)(smem + OFF_INFO);
  int* tcausal = (int*)(smem + OFF_INFO + 16);
  int* sbad = (int*)(smem + OFF_INFO + 24);

  pdl_launch_dependents();
  if (tid < PF_DEPTH) {
    mbar_init(&bars[tid], 1);
    sbad[tid] = 0;
  }
  fence_proxy_async();
  __syncthreads();
  pdl_wait();

  // this CTA's tiles
  const size_t head = (size_t)b * Hkv + kvh;
  // Lloyd-Max codebook levels of the kv head (used when a.codebook is set)
  const CbLevels cbk = cb_levels(a.rot.cb + (size_t)kvh * CB_WORDS);
  const CbLevels cbv = cb_levels(a.rot.cb + (size_t)(Hkv + kvh) * CB_WORDS);
  const int hist = cv.hist_lens[b];
  int pages = hist > 0 ? (hist + PAGE - 1) / PAGE : 0;
  if (pages > cv.max_pages_per_req) {  // inconsistent state: stay inside the page table
    if (tid == 0 && split == 0) record_error(cv.err, OSCAR_ERR_RANGE);
    pages = cv.max_pages_per_req;
  }
  int p0 = 0, n = 6;  // window: sink, ring quarters 0..3, chunk
  if (!win) {
    p0 = (int)((long long)split * pages / a.NS);
    n = (int)((long long)(split + 1) * pages / a.NS) - p0;
  }
  const int Lq = cv.seq_lens[b];
  const int nsink = Lq < SINK ? Lq : SINK;
  const int recent = Lq > SINK ? Lq - SINK - hist : 0;
  const int h0 = hist % RECENT;
  const int gbytes = cv.head_bytes;
  const int32_t* ptab = cv.page_table + (size_t)b * cv.max_pages_per_req;

  auto issue = [&](int i) {  // thread 0: bulk copy of history page p0 + i into slot i % PF_DEPTH
    const int slot = i % PF_DEPTH;
    const int pid = ptab[p0 + i];
    const bool ok = pid >= 0 && pid < cv.num_pages;
    sbad[slot] = ok ? 0 : 1;
    if (!ok) {
      record_error(cv.err, pid < 0 ? OSCAR_ERR_NO_PAGE : OSCAR_ERR_RANGE);
      mbar_expect_tx(&bars[slot], 0);
      return;
    }
    mbar_expect_tx(&bars[slot], (uint32_t)gbytes);
    bulk_g2s(smem + OFF_RAW + slot * RAW_SLOT, cv.pool + (size_t)pid * cv.page_bytes + (size_t)kvh * gbytes,
             (uint32_t)gbytes, &bars[slot]);
  };
  auto fill = [&](int i, int buf) {
    if (!win) {
      const int slot = i % PF_DEPTH;
      bool ok = mbar_wait(&bars[slot], (uint32_t)((i / PF_DEPTH) & 1));
      if (!ok) record_error(cv.err, OSCAR_ERR_TIMEOUT);
      ok = ok && !sbad[slot];
      const int pg = p0 + i;
      const int nv = pg == pages - 1 ? hist - pg * PAGE : PAGE;
      if (ok) {
        if (a.codebook)
          fill_int2<true>(smem, buf, smem + OFF_RAW + slot * RAW_SLOT, cv.g, nv, cbk, cbv);
        else
          fill_int2<false>(smem, buf, smem + OFF_RAW + slot * RAW_SLOT, cv.g, nv, cbk, cbv);
      }
      if (tid == 0) {
        tmask[buf] = ok ? low_mask(nv) : 0ull;
        tcausal[buf] = 0;
      }
      return;
    }
    uint64_t valid;
    const __nv_bfloat16 *Kb, *Vb;
    size_t stride = D;
    if (i == 0) {
      valid = low_mask(nsink);
      Kb = cv.sink_k + head * SINK * D;
      Vb = cv.sink_v + head * SINK * D;
    } else if (i <= 4) {
      const int s0 = 64 * (i - 1);
      const uint32_t lo = __ballot_sync(0xffffffffu, ((s0 + lane - h0 + RECENT) % RECENT) < recent);
      const uint32_t hi = __ballot_sync(0xffffffffu, ((s0 + 32 + lane - h0 + RECENT) % RECENT) < recent);
      valid = ((uint64_t)hi << 32) | lo;
      Kb = cv.ring_k + (head * RECENT + s0) * D;
      Vb = cv.ring_v + (head * RECENT + s0) * D;
    } else {
      valid = low_mask(a.T);
      stride = (size_t)Hkv * D;
      Kb = a.k + ((size_t)b * a.T * Hkv + kvh) * D;
      Vb = a.v + ((size_t)b * a.T * Hkv + kvh) * D;
    }
    fill_bf16(smem, buf, Kb, Vb, stride, valid);
    if (tid == 0) {
      tmask[buf] = valid;
      tcausal[buf] = i == 5;
    }
  };

  // query fragments of this warp's 16 rows (rotated for history, raw for the window)
  const int rbase = rt * PF_ROWS + 16 * warp;
  const __half* qb = a.qh + ((size_t)(win ? 1 : 0) * a.B * Hkv + bk) * RP * D + (size_t)rbase * D;
  uint32_t qa[8][4];
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) {
    const __half* q0 = qb + gid * D + 16 * ks + 2 * tig;
    qa[ks][0] = *(const uint32_t*)(q0);
    qa[ks][1] = *(const uint32_t*)(q0 + 8 * D);
    qa[ks][2] = *(const uint32_t*)(q0 + 8);
    qa[ks][3] = *(const uint32_t*)(q0 + 8 * D + 8);
  }
  const float al[2] = {a.alpha[(size_t)bk * RP + rbase + gid], a.alpha[(size_t)bk * RP + rbase + gid + 8]};
  const int trow[2] = {(rbase + gid) / G, (rbase + gid + 8) / G};
  RowState st;
#pragma unroll
  for (int j = 0; j < 16; ++j) st.o[j][0] = st.o[j][1] = st.o[j][2] = st.o[j][3] = 0.f;
  st.m[0] = st.m[1] = -1e30f;
  st.l[0] = st.l[1] = 0.f;
  const bool rows_live = rbase < R;

  if (!win && tid == 0)
    for (int i = 0; i < PF_DEPTH && i < n; ++i) issue(i);
  if (n > 0) fill(0, 0);
  __syncthreads();
  if (!win && tid == 0 && PF_DEPTH < n) issue(PF_DEPTH);
  const uint32_t tiles = (uint32_t)__cvta_generic_to_shared(smem + OFF_TILES);
  for (int i = 0; i < n; ++i) {
    const int buf = i & 1;
    if (i + 1 < n) fill(i + 1, buf ^ 1);
    const uint64_t mask = tmask[buf];
    if (mask && rows_live)
      tile_attend(st, qa, al, trow, tiles + buf * 2 * TILE_BYTES, tiles + buf * 2 * TILE_BYTES + TILE_BYTES,
                  mask, tcausal[buf] != 0, lane);
    __syncthreads();
    if (!win && tid == 0 && i + 1 + PF_DEPTH < n) issue(i + 1 + PF_DEPTH);
  }

  // partial records: m (log2 units), l, o (unnormalised)
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    st.l[h] += __shfl_xor_sync(0xffffffffu, st.l[h], 1);
    st.l[h] += __shfl_xor_sync(0xffffffffu, st.l[h], 2);
  }
  float* pbase = a.part + ((size_t)tile * (a.NS + 1) + split) * PF_ROWS * PART_STRIDE;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int ri = 16 * warp + gid + 8 * h;
    if (rt * PF_ROWS + ri >= R) continue;
    float* rec = pbase + (size_t)ri * PART_STRIDE;
    if (tig == 0) {
      rec[0] = st.m[h];
      rec[1] = st.l[h];
    }
#pragma unroll
    for (int j = 0; j < 16; ++j)
      *(float2*)(rec + PART_O + 8 * j + 2 * tig) = make_float2(st.o[j][2 * h], st.o[j][2 * h + 1]);
  }
}

constexpr int MROWS = 16;  // rows per merge CTA
constexpr int MERGE_SMEM = (D * D + MROWS * D) * 4;

// 16 rows of one tile by 256 threads: combine the history splits and the
// window partial, un-rotate the history part by R_V^T (staged in shared
// memory) and write out and lse.
__global__ void __launch_bounds__(256) prefill_merge_kernel(PrefillArgs a) {
  extern __shared__ __align__(16) float msm[];
  float* Rs = msm;         // [128][128] R_V^T: row k = column k of R_V
  float* xs = Rs + D * D;  // [16][128] combined history o'
  __shared__ float wsh[MROWS][PF_MAX_SPLITS + 1];
  __shared__ float linv[MROWS], lsev[MROWS];
  const CacheView& cv = a.cv;
  const int tile = blockIdx.x, bk = tile / a.RT, rt = tile % a.RT;
  const int b = bk / cv.Hkv, kvh = bk % cv.Hkv, G = cv.G;
  const int R = a.T * G, NS = a.NS, NSP = NS + 1;
  const int i0 = MROWS * blockIdx.y;
  const int tid = threadIdx.x, c = tid & 127, h = tid >> 7, warp = tid >> 5, lane = tid & 31;
  {  // the rotation table is written synchronously by oscar_set_rotation: load it before the wait
    const float4* Rg = (const float4*)(a.rot.RVt + (size_t)kvh * D * D);
    float4 rv[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) rv[j] = __ldg(Rg + tid + 256 * j);
#pragma unroll
    for (int j = 0; j < 16; ++j) ((float4*)Rs)[tid + 256 * j] = rv[j];
  }
  pdl_wait();
  pdl_launch_dependents();
  if (rt * PF_ROWS + i0 >= R) return;
  const float* base = a.part + (size_t)tile * NSP * PF_ROWS * PART_STRIDE;
  const size_t ss = (size_t)PF_ROWS * PART_STRIDE;  // between splits
  for (int j = warp; j < MROWS; j += 8) {  // softmax weights of the partials, warp per row
    const float* rb = base + (size_t)(i0 + j) * PART_STRIDE;
    float mv[3], lv[3], M = -INFINITY;
#pragma unroll
    for (int q = 0; q < 3; ++q) {
      const int s = lane + 32 * q;
      mv[q] = s < NSP ? rb[s * ss] : -INFINITY;
      lv[q] = s < NSP ? rb[s * ss + 1] : 0.f;
      M = fmaxf(M, mv[q]);
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float L = 0.f;
#pragma unroll
    for (int q = 0; q < 3; ++q) {
      const int s = lane + 32 * q;
      if (s < NSP) {
        const float w = ex2(mv[q] - M);
        wsh[j][s] = w;
        L += w * lv[q];
      }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
    if (lane == 0) {
      linv[j] = 1.f / L;
      lsev[j] = (M + log2f(L)) * LN2;
    }
  }
  __syncthreads();
  // thread (c, h): rows 8h .. 8h + 7; the loads of four splits at a time are in flight together
  float acc[8], ow[8];
  const float* cb = base + (size_t)(i0 + 8 * h) * PART_STRIDE + PART_O + c;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    acc[j] = 0.f;
    ow[j] = wsh[8 * h + j][NS] * cb[(size_t)j * PART_STRIDE + NS * ss];
  }
  for (int s = 0; s < NS; s += 4) {
    float v[4][8];
#pragma unroll
    for (int u = 0; u < 4; ++u)
#pragma unroll
      for (int j = 0; j < 8; ++j) v[u][j] = s + u < NS ? cb[(size_t)j * PART_STRIDE + (s + u) * ss] : 0.f;
#pragma unroll
    for (int u = 0; u < 4; ++u)
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[j] = fmaf(s + u < NS ? wsh[8 * h + j][s + u] : 0.f, v[u][j], acc[j]);
  }
#pragma unroll
  for (int j = 0; j < 8; ++j) xs[(8 * h + j) * D + c] = acc[j];
  __syncthreads();
  // o = o'·R_V^T: y_c = sum_k o'_k R_V[c][k]
  float y[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) y[j] = 0.f;
  const float* xh = xs + 8 * h * D;
#pragma unroll 2
  for (int k = 0; k < D; k += 4) {
    const float r0 = Rs[k * D + c], r1 = Rs[(k + 1) * D + c], r2 = Rs[(k + 2) * D + c], r3 = Rs[(k + 3) * D + c];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float4 x = *(const float4*)(xh + j * D + k);  // same address across the warp: one broadcast
      y[j] = fmaf(x.x, r0, fmaf(x.y, r1, fmaf(x.z, r2, fmaf(x.w, r3, y[j]))));
    }
  }
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int r = rt * PF_ROWS + i0 + 8 * h + j;
    if (r >= R) continue;
    const int lgG = __ffs(G) - 1;  // G is a power of two
    const size_t row = ((size_t)b * a.T + (r >> lgG)) * cv.Hq + kvh * G + (r & (G - 1));
    a.out[row * D + c] = __float2bfloat16_rn((y[j] + ow[j]) * linv[8 * h + j]);
    if (c == 0 && a.lse) a.lse[row] = lsev[8 * h + j];
  }
}


// ===================================================== tcgen05 attention
// The same work split and partial records as prefill_attn_kernel, on the
// fifth-generation tensor cores: S = Q·K^T and O += P·V as tcgen05.mma with
// M = 128 query rows; K and V^T in shared memory in the 128-byte-swizzled
// K-major layout; Q, S, P and O in tensor memory (Q and P are the A operands,
// so shared memory bandwidth goes to K and V only).  Warp roles:
//   warps 0-7  softmax, two warpgroups taking alternate pages, one query
//              row per thread (row = TMEM lane), each with its own O
//              accumulator (the two are merged like history splits)
//   warps 8-15 tile producers, two groups of four warps taking alternate
//              pages: dequantise a copied INT2 page (or convert BF16 window
//              rows) into the K and V^T tiles
//   warp 16    TMEM allocation and the tcgen05.mma issue (one thread)
//   warp 17    bulk copies of the INT2 pages into shared memory
// V^T carries 16 extra rows: a row of ones, whose O column accumulates the
// softmax row sum l from the same fp16 P the numerator uses, and 15 zero rows
// (N = 144, a multiple of 16).  O is rescaled lazily: only when a row maximum
// grows by more than LAZY (log2 units); until then P may reach 2^LAZY.
namespace tc {
constexpr int THREADS = 576;
constexpr int DQ0 = 256;    // first producer thread
constexpr int MMA_WARP = 16, TMA_WARP = 17;
constexpr int NKV = 4, NRAW = 8;
constexpr int VT_ROWS = 144;
constexpr int K_BYTES = 2 * PAGE * 128;     // two 64-dim regions of 64 tokens x 128 B
constexpr int VT_BYTES = VT_ROWS * 128;     // channels (+16) x 64 tokens
constexpr int KV_BYTES = K_BYTES + VT_BYTES;
constexpr int OFF_KV = 0;
constexpr int OFF_RAW = OFF_KV + NKV * KV_BYTES;
// (s2, z2) token-pair tables: [producer group][2][4 channel groups][32 token pairs]
constexpr int OFF_PAIRS = OFF_RAW + NRAW * RAW_SLOT;
constexpr int OFF_BAR = OFF_PAIRS + 2 * 2 * 4 * 32 * 8;
// barriers
constexpr int B_RAW_FULL = 0, B_RAW_EMPTY = B_RAW_FULL + NRAW, B_KV_FULL = B_RAW_EMPTY + NRAW,
              B_KV_EMPTY = B_KV_FULL + NKV,
              B_S_FULL = B_KV_EMPTY + NKV, B_P_FULL = B_S_FULL + 2, B_O_FINAL = B_P_FULL + 2,
              B_Q_FULL = B_O_FINAL + 2, B_DRAIN = B_Q_FULL + 1, NBARS = B_DRAIN + 1;
constexpr int OFF_INFO = OFF_BAR + NBARS * 8;  // per KV buffer {u64 mask, int causal, pad}; then misc ints
constexpr int OFF_MISC = OFF_INFO + NKV * 16;  // [0] tmem base, [1] abort, [2..2+NRAW) bad page
constexpr int SMEM_USED = OFF_MISC + 64;
constexpr int SMEM = SMEM_USED + 1024;  // slack to align the base to 1024 B
constexpr int TMEM_COLS = 512;
// O of warpgroup w at 160 w (144 used), Q at 320, S (and P) buffer j at 384 + 64 j
constexpr int O_COL0 = 0, Q_COL = 320, S_COL0 = 384;
constexpr float LAZY = 4.f;
constexpr uint32_t IDESC_S = (1u << 4) | ((uint32_t)(PAGE >> 3) << 17) | ((uint32_t)(PF_ROWS >> 4) << 24);
constexpr uint32_t IDESC_PV = (1u << 4) | ((uint32_t)(VT_ROWS >> 3) << 17) | ((uint32_t)(PF_ROWS >> 4) << 24);
static_assert(OFF_KV % 1024 == 0 && KV_BYTES % 1024 == 0 && K_BYTES % 1024 == 0, "swizzle atoms 1024-aligned");
static_assert(SMEM <= 227 * 1024, "shared memory");
static_assert(OFF_BAR % 8 == 0 && OFF_INFO % 8 == 0, "alignment");

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups
// 1024 B apart (the leading offset is unused for this layout).
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

__device__ __forceinline__ void mma_ts(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc));
}

__device__ __forceinline__ void commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(
                   (uint32_t)__cvta_generic_to_shared(bar))
               : "memory");
}

__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory"); }
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory"); }

__device__ __forceinline__ void arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"((uint32_t)__cvta_generic_to_shared(bar))
               : "memory");
}

#define OSCAR_R8(i) "=r"(r[i]), "=r"(r[i + 1]), "=r"(r[i + 2]), "=r"(r[i + 3]), "=r"(r[i + 4]), "=r"(r[i + 5]), \
                    "=r"(r[i + 6]), "=r"(r[i + 7])
// 32 consecutive 32-bit TMEM columns of this warp's 32 lanes, one lane per thread
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
      : OSCAR_R8(0), OSCAR_R8(8), OSCAR_R8(16), OSCAR_R8(24)
      : "r"(taddr));
}
#undef OSCAR_R8

#define OSCAR_W8(i) "r"(v[i]), "r"(v[i + 1]), "r"(v[i + 2]), "r"(v[i + 3]), "r"(v[i + 4]), "r"(v[i + 5]), \
                    "r"(v[i + 6]), "r"(v[i + 7])
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n" ::"r"(taddr),
      OSCAR_W8(0), OSCAR_W8(8), OSCAR_W8(16), OSCAR_W8(24)
      : "memory");
}
#undef OSCAR_W8
// One 32-bit TMEM column of this warp's 32 lanes (waits for it).
__device__ __forceinline__ float tmem_ld1(uint32_t taddr) {
  uint32_t r;
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];\n" : "=r"(r) : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;\n" : "+r"(r)::"memory");
  return __uint_as_float(r);
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory"); }

__device__ __forceinline__ uint32_t ex2_h2(uint32_t x) {
  uint32_t y;
  asm("ex2.approx.f16x2 %0, %1;\n" : "=r"(y) : "r"(x));
  return y;
}

// Bounded wait that also gives up as soon as another role has aborted.
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
  const uint32_t a = (uint32_t)__cvta_generic_to_shared(bar);
  for (int it = 0; it < (1 << 22); ++it) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(a), "r"(parity)
        : "memory");
    if (ok) return true;
    if ((it & 63) == 63 && *abort_flag) return false;
  }
  *abort_flag = 1;
  return false;
}

// The 128 threads of a producer group agree on a wait's outcome (named
// barrier `id`): all go on or all stop, so none is left behind at a later
// barrier.
__device__ __forceinline__ bool group_all(uint32_t id, bool ok) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %2, 0;\n bar.red.and.pred q, %1, 128, p;\n"
      " selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"(id), "r"((uint32_t)ok)
      : "memory");
  return r != 0;
}

// TMEM loads complete at tcgen05.wait::ld; the registers pass through the
// wait so that no use of them is scheduled before it.
#define OSCAR_P8(i) "+r"(r[i]), "+r"(r[i + 1]), "+r"(r[i + 2]), "+r"(r[i + 3]), "+r"(r[i + 4]), "+r"(r[i + 5]), \
                    "+r"(r[i + 6]), "+r"(r[i + 7])
__device__ __forceinline__ void tmem_ld_wait_regs(uint32_t (&r)[32]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;\n" : OSCAR_P8(0), OSCAR_P8(8), OSCAR_P8(16), OSCAR_P8(24)::"memory");
}
__device__ __forceinline__ void regs_after(uint32_t (&r)[32]) {
  asm volatile("" : OSCAR_P8(0), OSCAR_P8(8), OSCAR_P8(16), OSCAR_P8(24)::"memory");
}
#undef OSCAR_P8

// K chunk I (channels 64A + 8I .. +7) of token tr: words 2D + A, D = 0..3.
template <int I>
__device__ __forceinline__ void k_chunk(uint8_t* Kt, int tr, int A, uint32_t w0, uint32_t w1, uint32_t w2,
                                        uint32_t w3, uint32_t s2, uint32_t z2, bool ok) {
  uint4 v = make_uint4(0u, 0u, 0u, 0u);
  if (ok)
    v = make_uint4(hfma2u(codes_f16x2<I>(w0), s2, z2), hfma2u(codes_f16x2<I>(w1), s2, z2),
                   hfma2u(codes_f16x2<I>(w2), s2, z2), hfma2u(codes_f16x2<I>(w3), s2, z2));
  *(uint4*)(Kt + A * (PAGE * 128) + tr * 128 + ((I ^ (tr & 7)) << 4)) = v;
}

// V^T chunk I (token slots 8I .. 8I + 7) of channel ch: word T holds slots
// 8I + 2T and 8I + 2T + 1; pr = the channel group's (s, z) token-pair table.
template <int I, bool FULL>
__device__ __forceinline__ void v_chunk(uint8_t* Vt, int ch, uint4 w, const uint2* pr, int nv) {
  const uint4 p01 = *(const uint4*)(pr + 4 * I), p23 = *(const uint4*)(pr + 4 * I + 2);
  uint32_t v0 = hfma2u(codes_f16x2<I>(w.x), p01.x, p01.y);
  uint32_t v1 = hfma2u(codes_f16x2<I>(w.y), p01.z, p01.w);
  uint32_t v2 = hfma2u(codes_f16x2<I>(w.z), p23.x, p23.y);
  uint32_t v3 = hfma2u(codes_f16x2<I>(w.w), p23.z, p23.w);
  if (!FULL) {
    const int t0 = 8 * I;
    auto cut = [&](uint32_t v, int t) { return t + 1 < nv ? v : t < nv ? (v & 0xFFFFu) : 0u; };
    v0 = cut(v0, t0);
    v1 = cut(v1, t0 + 2);
    v2 = cut(v2, t0 + 4);
    v3 = cut(v3, t0 + 6);
  }
  *(uint4*)(Vt + ch * 128 + ((I ^ (ch & 7)) << 4)) = make_uint4(v0, v1, v2, v3);
}

// (s, z) of consecutive V token slots (2j, 2j + 1) per channel group, the
// operands of the V dequantisation, from one INT2 head block: threads
// t < 32 NG write entry [group t / 32][pair t % 32].
__device__ __forceinline__ void build_pairs(const uint8_t* raw, uint2* pairs, int NG, int t) {
  if (t < 32 * NG) {
    const uint32_t* vsz = (const uint32_t*)(raw + 4096 + 256 * NG);  // V (s, z) after the K (s, z)
    const int gp = t >> 5, j = t & 31;
    const uint32_t a = vsz[(2 * j) * NG + gp], b = vsz[(2 * j + 1) * NG + gp];
    pairs[gp * 32 + j] = make_uint2(prmt(a, b, 0x5410u), prmt(a, b, 0x7632u));
  }
}

// Dequantise one INT2 head block into K (two 64-channel regions) and V^T
// tiles with 16-byte stores, by the 128 threads of a producer group
// (t = 0..127): value = s·code + z with the group's fp16 scale and zero,
// rounded once to fp16.  g = 2^lg channels per group, NG = 128 / g groups;
// pairs = the block's build_pairs table; nv = valid tokens; FULL: all 64 are.
template <bool FULL>
__device__ __forceinline__ void dequant_page(uint8_t* Kt, uint8_t* Vt, const uint8_t* raw, const uint2* pairs,
                                             int lg, int NG, int nv, int t) {
  {  // K: token tr, chunks 4Ih .. 4Ih + 3 of both 64-channel halves
    const int tr = t & 63, Ih = t >> 6;
    const uint4 lo = *(const uint4*)(raw + tr * 32), hi = *(const uint4*)(raw + tr * 32 + 16);
    const uint32_t* ksz = (const uint32_t*)(raw + off_k_sz()) + tr * NG;
    const uint32_t sz0 = ksz[(32 * Ih) >> lg], sz1 = ksz[(64 + 32 * Ih) >> lg];
    const uint32_t s0 = prmt(sz0, sz0, 0x1010u), z0 = prmt(sz0, sz0, 0x3232u);
    const uint32_t s1 = prmt(sz1, sz1, 0x1010u), z1 = prmt(sz1, sz1, 0x3232u);
    const bool ok = FULL || tr < nv;
    if (Ih == 0) {
      k_chunk<0>(Kt, tr, 0, lo.x, lo.z, hi.x, hi.z, s0, z0, ok);
      k_chunk<0>(Kt, tr, 1, lo.y, lo.w, hi.y, hi.w, s1, z1, ok);
      k_chunk<1>(Kt, tr, 0, lo.x, lo.z, hi.x, hi.z, s0, z0, ok);
      k_chunk<1>(Kt, tr, 1, lo.y, lo.w, hi.y, hi.w, s1, z1, ok);
      k_chunk<2>(Kt, tr, 0, lo.x, lo.z, hi.x, hi.z, s0, z0, ok);
      k_chunk<2>(Kt, tr, 1, lo.y, lo.w, hi.y, hi.w, s1, z1, ok);
      k_chunk<3>(Kt, tr, 0, lo.x, lo.z, hi.x, hi.z, s0, z0, ok);
      k_chunk<3>(Kt, tr, 1, lo.y, lo.w, hi.y, hi.w, s1, z1, ok);
    } else {
      k_chunk<4>(Kt, tr, 0, lo.x, lo.z, hi.x, hi.z, s0, z0, ok);
      k_chunk<4>(Kt, tr, 1, lo.y, lo.w, hi.y, hi.w, s1, z1, ok);
      k_chunk<5>(Kt, tr, 0, lo.x, lo.z, hi.x, hi.z, s0, z0, ok);
      k_chunk<5>(Kt, tr, 1, lo.y, lo.w, hi.y, hi.w, s1, z1, ok);
      k_chunk<6>(Kt, tr, 0, lo.x, lo.z, hi.x, hi.z, s0, z0, ok);
      k_chunk<6>(Kt, tr, 1, lo.y, lo.w, hi.y, hi.w, s1, z1, ok);
      k_chunk<7>(Kt, tr, 0, lo.x, lo.z, hi.x, hi.z, s0, z0, ok);
      k_chunk<7>(Kt, tr, 1, lo.y, lo.w, hi.y, hi.w, s1, z1, ok);
    }
  }
  {  // V: channel t, all eight chunks
    const int ch = t;
    const uint4 w = *(const uint4*)(raw + 2048 + ch * 16);
    const uint2* pr = pairs + ((ch >> lg) << 5);
    v_chunk<0, FULL>(Vt, ch, w, pr, nv);
    v_chunk<1, FULL>(Vt, ch, w, pr, nv);
    v_chunk<2, FULL>(Vt, ch, w, pr, nv);
    v_chunk<3, FULL>(Vt, ch, w, pr, nv);
    v_chunk<4, FULL>(Vt, ch, w, pr, nv);
    v_chunk<5, FULL>(Vt, ch, w, pr, nv);
    v_chunk<6, FULL>(Vt, ch, w, pr, nv);
    v_chunk<7, FULL>(Vt, ch, w, pr, nv);
  }
}

// 64 BF16 tokens (row j at Kb + j·stride, Vb + j·stride) into the K and V^T
// tiles as fp16; rows with a clear bit in `valid` become zeros.
__device__ __forceinline__ void convert_bf16(uint8_t* Kt, uint8_t* Vt, const __nv_bfloat16* Kb,
                                             const __nv_bfloat16* Vb, size_t stride, uint64_t valid, int t) {
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int u = t + 128 * j, tok = u >> 4, c16 = u & 15;
    uint4 x = make_uint4(0u, 0u, 0u, 0u);
    if ((valid >> tok) & 1ull) x = *(const uint4*)(Kb + tok * stride + 8 * c16);
    const uint4 y = make_uint4(bf2_to_h2(x.x), bf2_to_h2(x.y), bf2_to_h2(x.z), bf2_to_h2(x.w));
    *(uint4*)(Kt + (c16 >> 3) * (PAGE * 128) + tok * 128 + (((c16 & 7) ^ (tok & 7)) << 4)) = y;
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int u = t + 128 * j, jp = u & 31, k8 = u >> 5;
    uint4 x0 = make_uint4(0u, 0u, 0u, 0u), x1 = x0;
    if ((valid >> (2 * jp)) & 1ull) x0 = *(const uint4*)(Vb + (2 * jp) * stride + 8 * k8);
    if ((valid >> (2 * jp + 1)) & 1ull) x1 = *(const uint4*)(Vb + (2 * jp + 1) * stride + 8 * k8);
    const uint32_t a[4] = {x0.x, x0.y, x0.z, x0.w}, b[4] = {x1.x, x1.y, x1.z, x1.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t lo = i & 1 ? (a[i >> 1] & 0xFFFF0000u) : (a[i >> 1] << 16);
      const uint32_t hi = i & 1 ? (b[i >> 1] & 0xFFFF0000u) : (b[i >> 1] << 16);
      *(uint32_t*)(Vt + (8 * k8 + i) * 128 + (((jp >> 2) ^ i) << 4) + 4 * (jp & 3)) =
          f2_to_h2(__uint_as_float(lo), __uint_as_float(hi));
    }
  }
}

// Window tile kinds: 0 sink, 1..4 ring quarters, 5 chunk.  Does [a, a + n)
// taken mod 256 meet [lo, lo + 64)?
__device__ __forceinline__ bool ring_meets(int a, int n, int lo) {
  if (n <= 0) return false;
  if (n >= RECENT) return true;
  const int e = a + n;
  if (a < lo + 64 && e > lo) return true;
  return e > RECENT && (e - RECENT) > lo;
}
}  // namespace tc

__global__ void __launch_bounds__(tc::THREADS, 1) prefill_tc_kernel(PrefillArgs a) {
  using namespace tc;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - ((uint32_t)__cvta_generic_to_shared(smem_raw) & 1023)) & 1023);
  const uint32_t sbase = (uint32_t)__cvta_generic_to_shared(smem);
  const CacheView& cv = a.cv;
  const int Hkv = cv.Hkv, G = cv.G;
  const int tile = blockIdx.x, bk = tile / a.RT, rt = tile % a.RT;
  const int b = bk / Hkv, kvh = bk % Hkv;
  const int split = blockIdx.y;
  const bool win = split == a.NS;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int R = a.T * G, RP = a.RT * PF_ROWS;
  uint64_t* bars = (uint64_t*)(smem + tc::OFF_BAR);
  uint8_t* info = smem + tc::OFF_INFO;
  int* misc = (int*)(smem + OFF_MISC);
  volatile int* abort_flag = misc + 1;

  pdl_launch_dependents();
  if (tid == 0) {
    for (int i = 0; i < NRAW; ++i) {
      mbar_init(&bars[B_RAW_FULL + i], 1);
      mbar_init(&bars[B_RAW_EMPTY + i], 4);  // the four warps of the page's producer group
    }
    for (int i = 0; i < NKV; ++i) {
      mbar_init(&bars[B_KV_FULL + i], 128);  // the page's producer group
      mbar_init(&bars[B_KV_EMPTY + i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars[B_S_FULL + i], 1);
      mbar_init(&bars[B_P_FULL + i], 4);
      mbar_init(&bars[B_O_FINAL + i], 1);
    }
    mbar_init(&bars[B_Q_FULL], 4);
    mbar_init(&bars[B_DRAIN], 1);
    misc[1] = 0;
    for (int i = 0; i < NRAW; ++i) misc[2 + i] = 0;
  }
  if (warp == MMA_WARP) {  // whole warp: allocate the tensor memory, publish its address
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(
                     (uint32_t)__cvta_generic_to_shared(&misc[0])),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
  }
  fence_proxy_async();
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = (uint32_t)misc[0];
  pdl_wait();

  // this CTA's tiles
  const size_t head = (size_t)b * Hkv + kvh;
  const int hist = cv.hist_lens[b];
  int pages = hist > 0 ? (hist + PAGE - 1) / PAGE : 0;
  if (pages > cv.max_pages_per_req) {
    if (tid == 0 && split == 0) record_error(cv.err, OSCAR_ERR_RANGE);
    pages = cv.max_pages_per_req;
  }
  const int Lq = cv.seq_lens[b];
  const int nsink = Lq < SINK ? Lq : SINK;
  const int recent = Lq > SINK ? Lq - SINK - hist : 0;
  const int h0 = ((hist % RECENT) + RECENT) % RECENT;
  int p0 = 0, n = 0;
  uint32_t kinds = 0;  // window: bit k set when tile kind k (0 sink, 1..4 ring quarters, 5 chunk) is present
  if (!win) {
    p0 = (int)((long long)split * pages / a.NS);
    n = (int)((long long)(split + 1) * pages / a.NS) - p0;
  } else {
    kinds = (nsink > 0 ? 1u : 0u) | (1u << 5);
#pragma unroll
    for (int q = 0; q < 4; ++q)
      if (ring_meets(h0, recent, 64 * q)) kinds |= 2u << q;
    n = __popc(kinds);
  }
  const int gbytes = cv.head_bytes;
  const int32_t* ptab = cv.page_table + (size_t)b * cv.max_pages_per_req;

  if (warp == MMA_WARP) {
    // ------------------------------------------------ tcgen05.mma issue
    if (lane == 0) {
      bool ok = wait_bar(&bars[B_Q_FULL], 0, abort_flag);
      for (int i = 0; ok && i <= n; ++i) {
        if (i < n) {  // S(i) = Q·K(i)^T into S buffer i % 2
          const int kb = i % NKV;
          if (!wait_bar(&bars[B_KV_FULL + kb], (i / NKV) & 1, abort_flag)) break;
          fence_after();
          const uint32_t kaddr = sbase + OFF_KV + kb * KV_BYTES;
          const uint32_t d = tmem + S_COL0 + 64 * (i & 1);
#pragma unroll
          for (int ks = 0; ks < 8; ++ks)
            mma_ts(d, tmem + Q_COL + 8 * ks, sdesc(kaddr + (ks >> 2) * (PAGE * 128) + (ks & 3) * 32), IDESC_S,
                   ks > 0);
          commit(&bars[B_S_FULL + (i & 1)]);
        }
        if (i >= 1) {  // O_w += P(j)·V(j), w = j % 2
          const int j = i - 1, kb = j % NKV, w = j & 1;
          if (!wait_bar(&bars[B_P_FULL + w], (j >> 1) & 1, abort_flag)) break;
          fence_after();
          const uint32_t vaddr = sbase + OFF_KV + kb * KV_BYTES + K_BYTES;
          const uint32_t pa = tmem + S_COL0 + 64 * w;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_ts(tmem + O_COL0 + 160 * w, pa + 8 * kk, sdesc(vaddr + kk * 32), IDESC_PV,
                   (j >= 2 || kk > 0) ? 1u : 0u);
          commit(&bars[B_KV_EMPTY + kb]);
          if (j >= n - 2) commit(&bars[B_O_FINAL + w]);
        }
      }
      // all issued MMAs complete before the tensor memory is released
      commit(&bars[B_DRAIN]);
      mbar_wait(&bars[B_DRAIN], 0);
    }
  } else if (warp == TMA_WARP) {
    // ------------------------------------------------ page copies (lane 0), page ids 32 at a time
    if (!win) {
      int issued = 0;
      int nxt = lane < n ? ptab[p0 + lane] : 0;
      for (int base = 0; base < n; base += 32) {
        const int mine = nxt;
        nxt = base + 32 + lane < n ? ptab[p0 + base + 32 + lane] : 0;
        const int cnt = n - base < 32 ? n - base : 32;
        int go = 1;
        for (int j = 0; j < cnt && go; ++j) {
          const int pid = __shfl_sync(0xffffffffu, mine, j);
          if (lane == 0) {
            const int i = base + j, slot = i % NRAW;
            if (i >= NRAW && !wait_bar(&bars[B_RAW_EMPTY + slot], ((i / NRAW) - 1) & 1, abort_flag)) {
              go = 0;
            } else {
              const bool ok = pid >= 0 && pid < cv.num_pages;
              misc[2 + slot] = ok ? 0 : 1;
              if (!ok) {
                record_error(cv.err, pid < 0 ? OSCAR_ERR_NO_PAGE : OSCAR_ERR_RANGE);
                mbar_expect_tx(&bars[B_RAW_FULL + slot], 0);
              } else {
                mbar_expect_tx(&bars[B_RAW_FULL + slot], (uint32_t)gbytes);
                bulk_g2s(smem + tc::OFF_RAW + slot * RAW_SLOT,
                         cv.pool + (size_t)pid * cv.page_bytes + (size_t)kvh * gbytes, (uint32_t)gbytes,
                         &bars[B_RAW_FULL + slot]);
              }
              issued = i + 1;
            }
          }
          go = __shfl_sync(0xffffffffu, go, 0);
        }
        if (!go) break;
      }
      // every copy this CTA started has landed before it exits
      if (lane == 0)
        for (int i = issued - NRAW < 0 ? 0 : issued - NRAW; i < issued; ++i)
          mbar_wait(&bars[B_RAW_FULL + i % NRAW], (i / NRAW) & 1);
    }
  } else if (tid >= DQ0) {
    // ------------------------------------------------ tile producers
    const int t = tid - DQ0;
    const int lg = 31 - __clz(cv.g), NG = D >> lg;
    // ones row (row sums) and zero rows below the 128 channels of every V^T
    // buffer (made visible to the tensor cores with the buffer's first tile)
    if (t < 128)
      for (int kb = 0; kb < NKV; ++kb) {
        const uint32_t v = (t < 8) ? 0x3C003C00u : 0u;
        *(uint4*)(smem + OFF_KV + kb * KV_BYTES + K_BYTES + 128 * 128 + 16 * t) = make_uint4(v, v, v, v);
      }
    const int pg = t >> 7, tq = t & 127;  // producer group (pages pg, pg + 2, ...), thread in it
    const uint32_t gbar = 5 + pg;         // the group's named barrier
    uint2* pairs0 = (uint2*)(smem + OFF_PAIRS) + pg * 256;
    int nn = n;
    // the (s, z) pair table of a page is built one page ahead (the first one here)
    if (!win && n > pg) {
      if (group_all(gbar, wait_bar(&bars[B_RAW_FULL + pg], 0, abort_flag)))
        build_pairs(smem + tc::OFF_RAW + pg * RAW_SLOT, pairs0, NG, tq);
      else
        nn = 0;
    }
    if (!win) {
      for (int k = 0;; ++k) {  // history pages pg, pg + 2, ...
        const int i = 2 * k + pg;
        if (i >= nn) break;
        const int kb = i % NKV, slot = i % NRAW;
        uint8_t* Kt = smem + OFF_KV + kb * KV_BYTES;
        bool okw = i < NKV || wait_bar(&bars[B_KV_EMPTY + kb], ((i / NKV) - 1) & 1, abort_flag);
        if (i + 2 < n) okw = okw && wait_bar(&bars[B_RAW_FULL + (i + 2) % NRAW], ((i + 2) / NRAW) & 1, abort_flag);
        // also: the group is done with its previous page and with this page's pair table
        if (!group_all(gbar, okw)) break;
        if (i + 2 < n)
          build_pairs(smem + tc::OFF_RAW + ((i + 2) % NRAW) * RAW_SLOT, pairs0 + ((k + 1) & 1) * 128, NG, tq);
        const int pgn = p0 + i;
        int nv = pgn == pages - 1 ? hist - pgn * PAGE : PAGE;
        if (misc[2 + slot]) nv = 0;
        const uint8_t* raw = smem + tc::OFF_RAW + slot * RAW_SLOT;
        if (nv == PAGE)
          dequant_page<true>(Kt, Kt + K_BYTES, raw, pairs0 + (k & 1) * 128, lg, NG, nv, tq);
        else
          dequant_page<false>(Kt, Kt + K_BYTES, raw, pairs0 + (k & 1) * 128, lg, NG, nv, tq);
        if (tq == 0) {
          *(uint64_t*)(info + kb * 16) = low_mask(nv);
          *(int*)(info + kb * 16 + 8) = 0;
        }
        fence_proxy_async();
        arrive(&bars[B_KV_FULL + kb]);
        __syncwarp();
        if (lane == 0) arrive(&bars[B_RAW_EMPTY + slot]);  // raw slot of page i free again
      }
    } else {
      for (int k = 0;; ++k) {  // window tiles pg, pg + 2, ...
        const int i = 2 * k + pg;
        if (i >= nn) break;
        const int kb = i % NKV;
        uint8_t* Kt = smem + OFF_KV + kb * KV_BYTES;
        const bool okw = i < NKV || wait_bar(&bars[B_KV_EMPTY + kb], ((i / NKV) - 1) & 1, abort_flag);
        if (!group_all(gbar, okw)) break;
        const int kind = __fns(kinds, 0, i + 1);  // the (i+1)-th present kind
        uint64_t mask;
        int causal = 0;
        const __nv_bfloat16 *Kb, *Vb;
        size_t stride = D;
        if (kind == 0) {
          mask = low_mask(nsink);
          Kb = cv.sink_k + head * SINK * D;
          Vb = cv.sink_v + head * SINK * D;
        } else if (kind <= 4) {
          const int s0 = 64 * (kind - 1);
          const uint32_t lo = __ballot_sync(0xffffffffu, ((s0 + lane - h0 + RECENT) % RECENT) < recent);
          const uint32_t hi = __ballot_sync(0xffffffffu, ((s0 + 32 + lane - h0 + RECENT) % RECENT) < recent);
          mask = ((uint64_t)hi << 32) | lo;
          Kb = cv.ring_k + (head * RECENT + s0) * D;
          Vb = cv.ring_v + (head * RECENT + s0) * D;
        } else {
          mask = low_mask(a.T);
          causal = 1;
          stride = (size_t)Hkv * D;
          Kb = a.k + ((size_t)b * a.T * Hkv + kvh) * D;
          Vb = a.v + ((size_t)b * a.T * Hkv + kvh) * D;
        }
        convert_bf16(Kt, Kt + K_BYTES, Kb, Vb, stride, mask, tq);
        if (tq == 0) {
          *(uint64_t*)(info + kb * 16) = mask;
          *(int*)(info + kb * 16 + 8) = causal;
        }
        fence_proxy_async();
        arrive(&bars[B_KV_FULL + kb]);
      }
    }
  } else {
    // ------------------------------------------------ softmax: warpgroup wg takes pages wg, wg + 2, ...
    const int wg = warp >> 2;
    const int row = tid & 127;  // = TMEM lane
    const int grow = rt * PF_ROWS + row;
    const float al = a.alpha[(size_t)bk * RP + grow];
    const int trow = grow / G;
    const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
    const uint32_t oa = tmem + lane_base + O_COL0 + 160 * wg;
    const uint32_t sa = tmem + lane_base + S_COL0 + 64 * wg;
    if (wg == 0) {  // this row of Q (rotated for history, raw for the window) -> TMEM
      const uint4* qrow = (const uint4*)(a.qh + ((size_t)(win ? 1 : 0) * a.B * Hkv + bk) * RP * D + (size_t)grow * D);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t v[32];
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint4 x = qrow[8 * h + c];
          v[4 * c] = x.x;
          v[4 * c + 1] = x.y;
          v[4 * c + 2] = x.z;
          v[4 * c + 3] = x.w;
        }
        tmem_st32(tmem + lane_base + Q_COL + 32 * h, v);
      }
      tmem_st_wait();
      fence_before();
      __syncwarp();
      if (lane == 0) arrive(&bars[B_Q_FULL]);
    }
    float m_run = -1e30f;
    bool ok = true;
    for (int k = 0;; ++k) {
      const int i = 2 * k + wg;
      if (i >= n) break;
      const int kb = i % NKV;
      if (!__all_sync(0xffffffffu, wait_bar(&bars[B_KV_FULL + kb], (i / NKV) & 1, abort_flag))) {
        ok = false;
        break;
      }
      const uint64_t mask = *(const uint64_t*)(info + kb * 16);
      const bool causal = *(const int*)(info + kb * 16 + 8) != 0;
      if (!__all_sync(0xffffffffu, wait_bar(&bars[B_S_FULL + wg], k & 1, abort_flag))) {
        ok = false;
        break;
      }
      fence_after();
      uint32_t r0[32], r1[32];
      tmem_ld32(sa, r0);
      tmem_ld32(sa + 32, r1);
      tmem_ld_wait_regs(r0);
      regs_after(r1);
      // raw logits (the row factor al > 0 is applied with the exponent)
      float x[64];
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        x[j] = __uint_as_float(r0[j]);
        x[32 + j] = __uint_as_float(r1[j]);
      }
      if (mask != ~0ull || causal) {
#pragma unroll
        for (int j = 0; j < 64; ++j)
          if (!((mask >> j) & 1ull) || (causal && j > trow)) x[j] = -INFINITY;
      }
      float m8[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) m8[j] = fmaxf(x[j], x[8 + j]);
#pragma unroll
      for (int j = 16; j < 64; ++j) m8[j & 7] = fmaxf(m8[j & 7], x[j]);
      const float mx = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                             fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7]))) * al;  // -inf stays -inf
      bool resc = false;
      float f = 1.f;
      if (k == 0) {
        m_run = fmaxf(m_run, mx);
      } else if (__any_sync(0xffffffffu, mx > m_run + LAZY)) {
        const float m_new = fmaxf(m_run, mx);
        f = ex2(m_run - m_new);
        m_run = m_new;
        resc = true;
      }
      {
        uint32_t p[32];
        const float nm = -m_run;
#pragma unroll
        for (int j = 0; j < 32; ++j) p[j] = ex2_h2(f2_to_h2(fmaf(x[2 * j], al, nm), fmaf(x[2 * j + 1], al, nm)));
        tmem_st32(sa, p);
      }
      if (resc) {
        // S(i) is complete, so is every MMA issued before it: O_wg holds P(i-2)·V(i-2)
#pragma unroll 1
        for (int c = 0; c < 160; c += 32) {  // columns 0..159 (the 144 in use and 16 unused)
          uint32_t v[32];
          tmem_ld32(oa + c, v);
          tmem_ld_wait_regs(v);
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = __float_as_uint(__uint_as_float(v[j]) * f);
          tmem_st32(oa + c, v);
          tmem_st_wait();
        }
      }
      tmem_st_wait();
      fence_before();
      __syncwarp();
      if (lane == 0) arrive(&bars[B_P_FULL + wg]);
    }
    // one partial record per CTA: m (log2 units), l, o (unnormalised).  With
    // two or more pages both warpgroups hold a partial: warpgroup 1 hands its
    // row to warpgroup 0 through the (then idle) first K/V buffers.
    float* rec = a.part + (((size_t)tile * (a.NS + 1) + split) * PF_ROWS + row) * PART_STRIDE;
    if (n >= 2) {
      float* xch = (float*)(smem + OFF_KV) + row * PART_STRIDE;
      ok = ok && __all_sync(0xffffffffu, wait_bar(&bars[B_O_FINAL], 0, abort_flag));
      ok = ok && __all_sync(0xffffffffu, wait_bar(&bars[B_O_FINAL + 1], 0, abort_flag));
      fence_after();
      if (wg == 1) {
#pragma unroll 1
        for (int c = 0; c < 128; c += 32) {
          uint32_t v[32];
          tmem_ld32(oa + c, v);
          tmem_ld_wait_regs(v);
#pragma unroll
          for (int j = 0; j < 32; j += 4)
            *(float4*)(xch + PART_O + c + j) = make_float4(__uint_as_float(v[j]), __uint_as_float(v[j + 1]),
                                                           __uint_as_float(v[j + 2]), __uint_as_float(v[j + 3]));
        }
        const float l1 = tmem_ld1(oa + 128);
        xch[0] = ok ? m_run : -1e30f;
        xch[1] = ok ? l1 : 0.f;
      }
      asm volatile("bar.sync 3, 256;\n" ::: "memory");  // the two softmax warpgroups
      if (wg == 0) {
        const float l0r = tmem_ld1(oa + 128);
        const float m0 = ok ? m_run : -1e30f, l0 = ok ? l0r : 0.f;
        const float m1 = xch[0], l1 = xch[1];
        const float M = fmaxf(m0, m1), w0 = ex2(m0 - M), w1 = ex2(m1 - M);
#pragma unroll 1
        for (int c = 0; c < 128; c += 32) {
          uint32_t v[32];
          tmem_ld32(oa + c, v);
          tmem_ld_wait_regs(v);
          if (grow < R) {
#pragma unroll
            for (int j = 0; j < 32; j += 4) {
              const float4 x1 = *(const float4*)(xch + PART_O + c + j);
              *(float4*)(rec + PART_O + c + j) =
                  make_float4(w0 * __uint_as_float(v[j]) + w1 * x1.x, w0 * __uint_as_float(v[j + 1]) + w1 * x1.y,
                              w0 * __uint_as_float(v[j + 2]) + w1 * x1.z, w0 * __uint_as_float(v[j + 3]) + w1 * x1.w);
            }
          }
        }
        if (grow < R) {
          rec[0] = M;
          rec[1] = w0 * l0 + w1 * l1;
        }
      }
    } else if (wg == 0) {
      if (ok && n == 1) ok = __all_sync(0xffffffffu, wait_bar(&bars[B_O_FINAL], 0, abort_flag));
      if (ok && n == 1) {
        fence_after();
#pragma unroll 1
        for (int c = 0; c < 128; c += 32) {
          uint32_t v[32];
          tmem_ld32(oa + c, v);
          tmem_ld_wait_regs(v);
          if (grow < R) {
#pragma unroll
            for (int j = 0; j < 32; j += 4)
              *(float4*)(rec + PART_O + c + j) = make_float4(__uint_as_float(v[j]), __uint_as_float(v[j + 1]),
                                                             __uint_as_float(v[j + 2]), __uint_as_float(v[j + 3]));
          }
        }
        const float l0 = tmem_ld1(oa + 128);
        if (grow < R) {
          rec[0] = m_run;
          rec[1] = l0;
        }
      } else if (grow < R) {  // no pages (or aborted): an empty partial
        rec[0] = -1e30f;
        rec[1] = 0.f;
        for (int j = 0; j < D; j += 4) *(float4*)(rec + PART_O + j) = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
  }
  fence_before();
  __syncthreads();
  if (tid == 0 && *abort_flag) record_error(cv.err, OSCAR_ERR_TIMEOUT);
  if (warp == MMA_WARP) {
    __syncwarp();
    fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(tmem), "r"(TMEM_COLS) : "memory");
  }
}

}  // namespace

PrefillScratch prefill_scratch_layout(int B, int Hkv, int G, int T, int NS) {
  const int RT = (T * G + PF_ROWS - 1) / PF_ROWS, RP = RT * PF_ROWS;
  PrefillScratch L;
  size_t off = 0;
  auto take = [&](size_t n) {
    const size_t o = off;
    off += (n + 255) & ~(size_t)255;
    return o;
  };
  L.off_qh = take((size_t)2 * B * Hkv * RP * D * sizeof(__half));
  L.off_alpha = take((size_t)B * Hkv * RP * sizeof(float));
  L.off_part = take((size_t)B * Hkv * RT * (NS + 1) * PF_ROWS * PART_STRIDE * sizeof(float));
  L.total = off;
  return L;
}

int prefill_max_splits(int B, int Hkv, int G, int T) {
  const long long tiles = (long long)B * Hkv * ((T * G + PF_ROWS - 1) / PF_ROWS);
  long long ns = 1024 / tiles;
  if (ns > PF_MAX_SPLITS) ns = PF_MAX_SPLITS;
  return ns < 1 ? 1 : (int)ns;
}

static cudaError_t ensure_prefill_smem() {
  static int l_attn[MAX_DEVICES], l_prep[MAX_DEVICES], l_merge[MAX_DEVICES], l_tc[MAX_DEVICES];
  cudaError_t e = raise_smem_limit(prefill_attn_kernel, l_attn, PF_SMEM);
  if (e == cudaSuccess) e = raise_smem_limit(prefill_prep_kernel, l_prep, PREP_SMEM);
  if (e == cudaSuccess) e = raise_smem_limit(prefill_merge_kernel, l_merge, MERGE_SMEM);
  if (e == cudaSuccess) e = raise_smem_limit(prefill_tc_kernel, l_tc, tc::SMEM);
  return e;
}

cudaError_t prefill_ctas_per_sm(int* n, int impl) {
  *n = 0;
  const cudaError_t e = ensure_prefill_smem();
  if (e != cudaSuccess) return e;
  if (impl == OSCAR_PREFILL_MMA_SYNC)
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(n, prefill_attn_kernel, PF_THREADS, PF_SMEM);
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(n, prefill_tc_kernel, tc::THREADS, tc::SMEM);
}

cudaError_t launch_prefill(const PrefillArgs& a, cudaStream_t st, Profiler* prof) {
  cudaError_t e = ensure_prefill_smem();
  if (e != cudaSuccess) return e;
  const int tiles = a.B * a.cv.Hkv * a.RT;
  const PrefillArgs& b = a;
  prof_begin(prof, OSCAR_KERNEL_PREFILL_PREP, st);
  e = launch_pdl(prefill_prep_kernel, dim3(a.B * a.cv.Hkv, a.RT * (PF_ROWS / PREP_ROWS)), dim3(256), PREP_SMEM, st,
                 b);
  prof_end(prof, OSCAR_KERNEL_PREFILL_PREP, st);
  if (e != cudaSuccess) return e;
  prof_begin(prof, OSCAR_KERNEL_PREFILL_ATTN, st);
  if (a.impl == OSCAR_PREFILL_MMA_SYNC)
    e = launch_pdl(prefill_attn_kernel, dim3(tiles, a.NS + 1), dim3(PF_THREADS), PF_SMEM, st, b);
  else
    e = launch_pdl(prefill_tc_kernel, dim3(tiles, a.NS + 1), dim3(tc::THREADS), tc::SMEM, st, b);
  prof_end(prof, OSCAR_KERNEL_PREFILL_ATTN, st);
  if (e != cudaSuccess) return e;
  prof_begin(prof, OSCAR_KERNEL_PREFILL_MERGE, st);
  e = launch_pdl(prefill_merge_kernel, dim3(tiles, PF_ROWS / MROWS), dim3(256), MERGE_SMEM, st, b);
  prof_end(prof, OSCAR_KERNEL_PREFILL_MERGE, st);
  return e;
}

}  // namespace oscar
