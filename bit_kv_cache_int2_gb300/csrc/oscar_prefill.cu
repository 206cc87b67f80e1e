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
constexpr int MERGE_ROWS = 8;
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

// ------------------------------------------------------------ tile filling
// K tile: row = token (256 B), 16-byte chunk j of row t stored at j ^ (t & 7).
// V^T tile: row = channel (128 B), chunk j of row c stored at j ^ (c & 7).
// Tokens outside the tile's valid set are written as zeros.

// Dequantise one INT2 head block (raw, in shared memory) into the K and V^T
// tiles: value = s·code + z with the group's fp16 scale and zero, rounded
// once to fp16.  nv = valid tokens (rows 0..nv-1).
template <int I>
__device__ __forceinline__ void k_store(uint8_t* Kt, int tr, int A, int dq, uint32_t w, uint32_t s2,
                                        uint32_t z2, bool ok) {
  const uint32_t val = ok ? hfma2u(codes_f16x2<I>(w), s2, z2) : 0u;
  *(uint32_t*)(Kt + tr * 256 + ((((8 * A + I) ^ (tr & 7))) << 4) + 4 * dq) = val;
}

template <int I>
__device__ __forceinline__ void v_store(uint8_t* Vt, int ch, int T4, uint32_t w, const uint32_t* vsz,
                                        int NG, int grp, int nv) {
  const int t = 8 * I + 2 * T4;  // token slot of the low half; t + 1 in the high half
  const uint32_t a = vsz[t * NG + grp], b = vsz[(t + 1) * NG + grp];
  uint32_t val = hfma2u(codes_f16x2<I>(w), prmt(a, b, 0x5410u), prmt(a, b, 0x7632u));
  if (t + 1 >= nv) val = t < nv ? (val & 0xFFFFu) : 0u;
  *(uint32_t*)(Vt + ch * 128 + (((I ^ (ch & 7))) << 4) + 4 * T4) = val;
}

__device__ __forceinline__ void fill_int2(uint8_t* smem, int buf, const uint8_t* raw, int g, int nv) {
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
      k_store<0>(Kt, tr, A, dq, w, s0, z0, ok);
      k_store<1>(Kt, tr, A, dq, w, s0, z0, ok);
      k_store<2>(Kt, tr, A, dq, w, s0, z0, ok);
      k_store<3>(Kt, tr, A, dq, w, s0, z0, ok);
      k_store<4>(Kt, tr, A, dq, w, s1, z1, ok);
      k_store<5>(Kt, tr, A, dq, w, s1, z1, ok);
      k_store<6>(Kt, tr, A, dq, w, s1, z1, ok);
      k_store<7>(Kt, tr, A, dq, w, s1, z1, ok);
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
      v_store<0>(Vt, ch, T4, w, vsz, NG, grp, nv);
      v_store<1>(Vt, ch, T4, w, vsz, NG, grp, nv);
      v_store<2>(Vt, ch, T4, w, vsz, NG, grp, nv);
      v_store<3>(Vt, ch, T4, w, vsz, NG, grp, nv);
      v_store<4>(Vt, ch, T4, w, vsz, NG, grp, nv);
      v_store<5>(Vt, ch, T4, w, vsz, NG, grp, nv);
      v_store<6>(Vt, ch, T4, w, vsz, NG, grp, nv);
      v_store<7>(Vt, ch, T4, w, vsz, NG, grp, nv);
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
__global__ void __launch_bounds__(128) prefill_prep_kernel(PrefillArgs a) {
  __shared__ float xs[8][D];
  __shared__ float nrm[8];
  const CacheView& cv = a.cv;
  const int bk = blockIdx.x, b = bk / cv.Hkv, kvh = bk % cv.Hkv, G = cv.G;
  const int R = a.T * G, RP = a.RT * PF_ROWS, r0 = 8 * blockIdx.y;
  const int c = threadIdx.x, w = c >> 5, lane = c & 31;
  const float* Rk = a.rot.R_K + (size_t)kvh * D * D + c;
  pdl_wait();
  pdl_launch_dependents();
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int r = r0 + j;
    xs[j][c] = r < R ? __bfloat162float(a.q[(((size_t)b * a.T + r / G) * cv.Hq + kvh * G + r % G) * D + c])
                     : 0.f;
  }
  __syncthreads();
#pragma unroll
  for (int jj = 0; jj < 2; ++jj) {
    const int j = 2 * w + jj;
    float sq = 0.f;
#pragma unroll
    for (int k = 0; k < 4; ++k) sq = fmaf(xs[j][lane + 32 * k], xs[j][lane + 32 * k], sq);
#pragma unroll
    for (int o = 16; o; o >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, o);
    if (lane == 0) nrm[j] = sqrtf(sq);
  }
  __syncthreads();
  float acc[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) acc[j] = 0.f;
#pragma unroll 4
  for (int k = 0; k < D; ++k) {
    const float rk = __ldg(Rk + (size_t)k * D);
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j] = fmaf(xs[j][k], rk, acc[j]);
  }
  const size_t vstride = (size_t)a.B * cv.Hkv * RP * D;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int r = r0 + j;
    // |q'_c| and |q_c| are both at most |q| (R_K is orthogonal): 2^-sigma
    // brings them below 2^14 in fp16
    int ex = 0;
    frexpf(nrm[j], &ex);
    const int sig = nrm[j] > 0.f ? ex - 14 : 0;
    const size_t e = ((size_t)bk * RP + r) * D + c;
    a.qh[e] = __float2half_rn(ldexpf(acc[j], -sig));
    a.qh[vstride + e] = __float2half_rn(ldexpf(xs[j][c], -sig));
    if (c == 0) a.alpha[(size_t)bk * RP + r] = ldexpf(1.f, sig) * LOG2E * INV_SQRT_D;
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
      if (ok) fill_int2(smem, buf, smem + OFF_RAW + slot * RAW_SLOT, cv.g, nv);
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

__global__ void __launch_bounds__(128) prefill_merge_kernel(PrefillArgs a) {
  __shared__ float xs[MERGE_ROWS][D];
  __shared__ float wsh[MERGE_ROWS][PF_MAX_SPLITS + 1];
  __shared__ float linv[MERGE_ROWS], lsev[MERGE_ROWS];
  const CacheView& cv = a.cv;
  const int tile = blockIdx.x, bk = tile / a.RT, rt = tile % a.RT;
  const int b = bk / cv.Hkv, kvh = bk % cv.Hkv, G = cv.G;
  const int R = a.T * G, NS = a.NS, NSP = NS + 1;
  const int i0 = MERGE_ROWS * blockIdx.y;
  const int c = threadIdx.x, warp = c >> 5, lane = c & 31;
  pdl_wait();
  pdl_launch_dependents();
  if (rt * PF_ROWS + i0 >= R) return;
  const float* base = a.part + (size_t)tile * NSP * PF_ROWS * PART_STRIDE;
  const size_t ss = (size_t)PF_ROWS * PART_STRIDE;  // between splits
  for (int j = warp; j < MERGE_ROWS; j += 4) {
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
  float ow[MERGE_ROWS];
#pragma unroll
  for (int j = 0; j < MERGE_ROWS; ++j) {
    const float* rb = base + (size_t)(i0 + j) * PART_STRIDE + PART_O + c;
    float acc = 0.f;
    for (int s = 0; s < NS; ++s) acc = fmaf(wsh[j][s], rb[s * ss], acc);
    xs[j][c] = acc;
    ow[j] = wsh[j][NS] * rb[NS * ss];
  }
  __syncthreads();
  // o = o'·R_V^T: y_c = sum_k o'_k R_V[c][k], RVt row k = column k of R_V^T
  const float* Rt = a.rot.RVt + (size_t)kvh * D * D + c;
  float y[MERGE_ROWS];
#pragma unroll
  for (int j = 0; j < MERGE_ROWS; ++j) y[j] = 0.f;
#pragma unroll 4
  for (int k = 0; k < D; ++k) {
    const float r = __ldg(Rt + (size_t)k * D);
#pragma unroll
    for (int j = 0; j < MERGE_ROWS; ++j) y[j] = fmaf(xs[j][k], r, y[j]);
  }
#pragma unroll
  for (int j = 0; j < MERGE_ROWS; ++j) {
    const int r = rt * PF_ROWS + i0 + j;
    if (r >= R) continue;
    const size_t row = ((size_t)b * a.T + r / G) * cv.Hq + kvh * G + r % G;
    a.out[row * D + c] = __float2bfloat16_rn((y[j] + ow[j]) * linv[j]);
    if (c == 0 && a.lse) a.lse[row] = lsev[j];
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
  static int done = 0;  // per process; the attribute is per device function
  if (done) return cudaSuccess;
  const cudaError_t e =
      cudaFuncSetAttribute(prefill_attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, PF_SMEM);
  if (e == cudaSuccess) done = 1;
  return e;
}

cudaError_t prefill_ctas_per_sm(int* n) {
  *n = 0;
  const cudaError_t e = ensure_prefill_smem();
  if (e != cudaSuccess) return e;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(n, prefill_attn_kernel, PF_THREADS, PF_SMEM);
}

cudaError_t launch_prefill(const PrefillArgs& a, cudaStream_t st, Profiler* prof) {
  cudaError_t e = ensure_prefill_smem();
  if (e != cudaSuccess) return e;
  const int tiles = a.B * a.cv.Hkv * a.RT;
  prof_begin(prof, OSCAR_KERNEL_PREFILL_PREP, st);
  e = launch_pdl(prefill_prep_kernel, dim3(a.B * a.cv.Hkv, a.RT * (PF_ROWS / 8)), dim3(128), 0, st, a);
  prof_end(prof, OSCAR_KERNEL_PREFILL_PREP, st);
  if (e != cudaSuccess) return e;
  prof_begin(prof, OSCAR_KERNEL_PREFILL_ATTN, st);
  e = launch_pdl(prefill_attn_kernel, dim3(tiles, a.NS + 1), dim3(PF_THREADS), PF_SMEM, st, a);
  prof_end(prof, OSCAR_KERNEL_PREFILL_ATTN, st);
  if (e != cudaSuccess) return e;
  prof_begin(prof, OSCAR_KERNEL_PREFILL_MERGE, st);
  e = launch_pdl(prefill_merge_kernel, dim3(tiles, PF_ROWS / MERGE_ROWS), dim3(128), 0, st, a);
  prof_end(prof, OSCAR_KERNEL_PREFILL_MERGE, st);
  return e;
}

}  // namespace oscar
