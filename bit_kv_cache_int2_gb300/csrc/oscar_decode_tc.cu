// INT2 history decode on the fifth-generation tensor cores (sm_103a).
//
// The same computation as decode_kernel (oscar_decode.cu) -- the decode
// paragraph under the pipeline figure "从离线校准到在线推理的pipeline" of
// "超越TurboQuant：Together AI把2-bit KV Cache推向真实服务": the INT2 history is
// unpacked, dequantised with its scale / zero point and accumulated in
// floating point, the BF16 sink/recent segment is attended separately, and
// the parts are merged by online softmax (merge_kernel) -- laid out for
// tcgen05 and tensor memory instead of mma.sync fragments.
//
// One persistent CTA per SM takes a contiguous, equal share of the work
// (balanced partition, oscar_internal.cuh).  History is processed in tiles of
// two pages (128 tokens) of one kv head.  Warp roles:
//   warps 0-3  token warps: thread r = tile row r (page r / 64, token r % 64).
//              Unpack the token's 128 K codes straight into tensor memory as
//              the A operand of S = K·q'^T (M = 128 tokens); read its logits
//              back (one row per thread), apply the K scale / zero point,
//              the online softmax, and write P·s (the A = V^T product's
//              B operand) into shared memory.  They also attend the BF16
//              window chunks of the CTA (mma.sync, before the history starts).
//   warps 4-7  channel warps: thread c = rotated channel c.  Unpack the
//              channel's 128 V codes of the tile into tensor memory as the A
//              operand of O^T += V^T·(P·s) (M = 128 channels); at the end of an
//              item read O back, add the zero-point term and write the
//              item's partial record.
//   warp 8     page copies (one bulk copy per page and kv head) into a ring
//              of shared-memory stages.
//   warp 9     tensor-memory allocation and the tcgen05.mma issue.
// A code c at bit pair I of a 16-bit half becomes the fp16 subnormal
// c * 2^(E(I) - 24) with one AND (E = 4, 6 or 8, the 2-bit field's position),
// so the products carry no offset; the 2^(8 - E) and 2^(7 - E) factors go
// into the B operands (q' in shared memory, P·s per token).  Scale and zero
// point are applied in fp32 outside the products: per token for the logits,
// per group column for the output.
#include "oscar_internal.cuh"
#include "oscar_window.cuh"

namespace oscar {
namespace {
namespace dtc {

constexpr int THREADS = 320;
constexpr int CW = 4;     // token warps 0..3, channel warps 4..7
constexpr int LD_WARP = 8, MMA_WARP = 9;
constexpr int NST = 6;    // page-pair stages
constexpr int TMEM_COLS = 512;
constexpr int AK_COL = 0;    // A operand of S, 2 buffers x 64 columns (128 fp16 channels per row)
constexpr int AV_COL = 128;  // A operand of O^T, 2 buffers x 64 columns (128 fp16 tokens per row)
constexpr int D_COL = 256;   // S, 2 buffers x NQ columns; O follows at D_COL + 2 NQ, 2 buffers
constexpr float TAU = 4.f;   // lazy rescale: P may reach 2^TAU before the running maximum moves
constexpr int MAXNQ = 32;    // NQ = G * (128 / g) columns, rounded up to 16 (at most 32)
constexpr int WCH = 8;       // weight of a BF16 window chunk in page units (balanced partition)

// barriers (index into the mbarrier array)
constexpr int B_ST_FULL = 0, B_ST_EMPTY = B_ST_FULL + NST, B_AK_FULL = B_ST_EMPTY + NST, B_AV_FULL = B_AK_FULL + 2,
              B_D_FULL = B_AV_FULL + 2, B_D_EMPTY = B_D_FULL + 2, B_B_FULL = B_D_EMPTY + 2,
              B_SV_DONE = B_B_FULL + 2, B_O_FULL = B_SV_DONE + 2, B_O_EMPTY = B_O_FULL + 2,
              B_STATS = B_O_EMPTY + 2, B_DRAIN = B_STATS + 2, NBARS = B_DRAIN + 1;

// Shared memory: stages (NST x 2 head blocks), B operands (q' and P·s, two
// of each, 128-byte-swizzled K-major, 1024-aligned), window scratch, tables.
struct Layout {
  int stage_bytes, off_stage, off_bq, off_bsv, bop_bytes, off_win, off_kc, off_stats, off_red, off_bar, off_flags,
      off_misc, off_pre, total;
};

__host__ __device__ inline Layout layout(int head_bytes, int B) {
  Layout L;
  L.stage_bytes = (2 * head_bytes + 127) & ~127;
  int o = 0;
  L.off_stage = o;
  o += NST * L.stage_bytes;
  o = (o + 1023) & ~1023;
  L.bop_bytes = MAXNQ * 256;  // NQ rows x 128 fp16
  L.off_bq = o;
  o += 2 * L.bop_bytes;
  L.off_bsv = o;
  o += 2 * L.bop_bytes;
  L.off_win = o;  // window chunk: per-warp m, l [4][MAX_G] each and o [4][MAX_G][128]
  o += 2 * 4 * MAX_G * 4 + 4 * MAX_G * D * 4;
  L.off_kc = o;  // per history item parity: ka[MAX_G], kg[MAX_G][4]
  o += 2 * (MAX_G + MAX_G * 4) * 4;
  L.off_stats = o;  // per item parity: m[MAX_G], l[MAX_G], zs[MAX_G][4]
  o += 2 * (2 * MAX_G + MAX_G * 4) * 4;
  L.off_red = o;  // token-warp exchange: [4 warps][MAX_G + MAX_G * 4] floats
  o += 4 * (MAX_G + MAX_G * 4) * 4;
  L.off_bar = (o + 7) & ~7;
  o = L.off_bar + NBARS * 8;
  L.off_flags = o;  // per stage: bit 0 page A copied, bit 1 page B copied
  o += NST * 4;
  L.off_misc = o;  // [0] tmem base, [1] abort
  o += 16;
  L.off_pre = (o + 7) & ~7;
  o = L.off_pre + (B + 1) * 8;
  L.total = o + 1024;  // slack to align the base to 1024 bytes
  return L;
}

__host__ __device__ constexpr uint32_t idesc(int nq) {
  // kind::f16: fp16 A and B, fp32 D, both K-major; N = nq, M = 128
  return (1u << 4) | ((uint32_t)(nq >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
}

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups
// 1024 B apart (the leading offset is unused for this layout).
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// Byte offset of element (row n, k) of an NQ-row, 128-column fp16 operand in
// the 128-byte-swizzled K-major layout: two 64-column regions of NQ rows.
__device__ __forceinline__ int bop_offset(int nq, int n, int k) {
  const int kk = k & 63;
  return (k >> 6) * (nq * 128) + n * 128 + (((kk >> 3) ^ (n & 7)) << 4) + (kk & 7) * 2;
}

__device__ __forceinline__ void mma_ts(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t id, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d),
      "r"(a_tmem), "l"(b), "r"(id), "r"(acc));
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
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n"
      : OSCAR_R8(0), OSCAR_R8(8)
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
      : OSCAR_R8(0), OSCAR_R8(8), OSCAR_R8(16), OSCAR_R8(24)
      : "r"(taddr));
}
#undef OSCAR_R8
#define OSCAR_P8(i) "+r"(r[i]), "+r"(r[i + 1]), "+r"(r[i + 2]), "+r"(r[i + 3]), "+r"(r[i + 4]), "+r"(r[i + 5]), \
                    "+r"(r[i + 6]), "+r"(r[i + 7])
// TMEM loads complete at tcgen05.wait::ld; the registers pass through the
// wait so that no use of them is scheduled before it.
__device__ __forceinline__ void tmem_ld_wait16(uint32_t* r) {
  asm volatile("tcgen05.wait::ld.sync.aligned;\n" : OSCAR_P8(0), OSCAR_P8(8)::"memory");
}
__device__ __forceinline__ void tmem_ld_wait32(uint32_t* r) {
  asm volatile("tcgen05.wait::ld.sync.aligned;\n" : OSCAR_P8(0), OSCAR_P8(8), OSCAR_P8(16), OSCAR_P8(24)::"memory");
}
#undef OSCAR_P8
#define OSCAR_W8(i) "r"(v[i]), "r"(v[i + 1]), "r"(v[i + 2]), "r"(v[i + 3]), "r"(v[i + 4]), "r"(v[i + 5]), \
                    "r"(v[i + 6]), "r"(v[i + 7])
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};\n" ::"r"(
          taddr),
      OSCAR_W8(0), OSCAR_W8(8)
      : "memory");
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n" ::"r"(taddr),
      OSCAR_W8(0), OSCAR_W8(8), OSCAR_W8(16), OSCAR_W8(24)
      : "memory");
}
#undef OSCAR_W8
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory"); }

// The 8 code pairs of word w into v[0..7] (v[I] = pair I).
__device__ __forceinline__ void word_codes(uint32_t w, uint32_t* v) {
  v[0] = code_sub<0>(w);
  v[1] = code_sub<1>(w);
  v[2] = code_sub<2>(w);
  v[3] = code_sub<3>(w);
  v[4] = code_sub<4>(w);
  v[5] = code_sub<5>(w);
  v[6] = code_sub<6>(w);
  v[7] = code_sub<7>(w);
}

// Bounded wait that gives up early once another role has aborted; a timeout
// sets the abort flag and records the error.
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, volatile int* abort_flag, int* err) {
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
  record_error(err, OSCAR_ERR_TIMEOUT);
  return false;
}

// The 128 token-warp threads agree: true when `pred` holds in any of them
// (named barrier 1).
__device__ __forceinline__ bool tw_any(bool pred) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.or.pred q, 1, 128, p;\n"
      " selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"((uint32_t)pred)
      : "memory");
  return r != 0;
}
__device__ __forceinline__ void tw_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// A history item: pages [p0, p1) of (b, kvh).
struct Item {
  int b, kvh, p0, p1, slot;
};

// Walks the segments that overlap [lo, hi) and calls f(b, kvh, seg_start, P,
// mask, wb) for each, in order.
template <typename F>
__device__ __forceinline__ void for_segments(const CacheView& cv, int B, const long long* pre, long long lo,
                                             long long hi, int wch, F&& f) {
  if (lo >= hi) return;
  int b = balanced_request(pre, B, lo);
  for (; b < B; ++b) {
    if (pre[b] >= hi) return;
    const int H = cv.hist_lens[b], Lq = cv.seq_lens[b];
    const int P = H > 0 ? (H + PAGE - 1) / PAGE : 0;
    const unsigned mask = window_chunk_mask(Lq, H);
    const long long wb = P + (long long)wch * __popc(mask);
    if (wb == 0) continue;
    int kvh = pre[b] < lo ? (int)((lo - pre[b]) / wb) : 0;
    for (; kvh < cv.Hkv; ++kvh) {
      const long long seg = pre[b] + (long long)kvh * wb;
      if (seg >= hi) return;
      f(b, kvh, seg, P, mask);
    }
  }
}

// The CTA's history items, in order; returns their number (calls g(item, index)).
template <typename F>
__device__ __forceinline__ int for_hist_items(const CacheView& cv, int B, const long long* pre, long long lo,
                                              long long hi, int wch, int cta, F&& g) {
  int n = 0;
  for_segments(cv, B, pre, lo, hi, wch, [&](int b, int kvh, long long seg, int P, unsigned) {
    const long long a = lo > seg ? lo : seg;
    const long long e = hi < seg + P ? hi : seg + P;
    if (a < e) {
      Item it;
      it.b = b;
      it.kvh = kvh;
      it.p0 = (int)(a - seg);
      it.p1 = (int)(e - seg);
      it.slot = cta + b * cv.Hkv + kvh;
      g(it, n);
      ++n;
    }
  });
  return n;
}

// Kernel parameters derived once per CTA.
struct Ctx {
  uint8_t* smem;
  uint32_t sbase;
  uint64_t* bars;
  volatile int* abort_flag;
  int* err;
  Layout L;
  int nq;
};

}  // namespace dtc

using namespace dtc;

// ------------------------------------------------------------ token warps
// Window chunk c of (b, kvh) on mma.sync (BF16, unrotated q): warp w takes
// tokens 16w .. 16w + 15 of the chunk; the four warps' states are combined
// into the chunk's partial record.
__device__ __forceinline__ void tw_window_chunk(const DecodeArgs& a, const Ctx& X, int b, int kvh, int c, int slot) {
  const CacheView& cv = a.cv;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gid = lane >> 2, tq = lane & 3;
  const int G = cv.G, Hkv = cv.Hkv;
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
  const int Lq = cv.seq_lens[b], hist = cv.hist_lens[b];
  const int nsink = Lq < SINK ? Lq : SINK;
  const int recent = Lq > SINK ? Lq - SINK - hist : 0;
  const int h0 = hist % RECENT;
  uint64_t valid = 0;
  const __nv_bfloat16 *Kb, *Vb;
  if (c == 0) {
    valid = nsink >= 64 ? ~0ull : ((1ull << nsink) - 1ull);
    Kb = cv.sink_k + head * SINK * D;
    Vb = cv.sink_v + head * SINK * D;
  } else {
    const int s0 = 64 * (c - 1);
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int t = lane + 32 * half;
      const bool v = ((s0 + t - h0 + RECENT) % RECENT) < recent;
      valid |= (uint64_t)__ballot_sync(0xffffffffu, v) << (32 * half);
    }
    Kb = cv.ring_k + (head * RECENT + s0) * D;
    Vb = cv.ring_v + (head * RECENT + s0) * D;
  }
  if ((valid >> (16 * warp)) & 0xFFFFull) bf16_span_mma<false>(S, Kb, Vb, valid, lane, warp, 1);
#pragma unroll
  for (int hc = 0; hc < 2; ++hc) {
    S.l[hc] += __shfl_xor_sync(0xffffffffu, S.l[hc], 4);
    S.l[hc] += __shfl_xor_sync(0xffffffffu, S.l[hc], 8);
    S.l[hc] += __shfl_xor_sync(0xffffffffu, S.l[hc], 16);
  }
  float* wm = (float*)(X.smem + X.L.off_win);
  float* wl = wm + 4 * MAX_G;
  float* wo = wl + 4 * MAX_G;
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
  tw_sync();
  const int ch = threadIdx.x;  // one channel per token-warp thread
  for (int n = 0; n < G; ++n) {
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < 4; ++w) M = fmaxf(M, wm[w * MAX_G + n]);
    float Ls = 0.f, O = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const float mw = wm[w * MAX_G + n];
        const float f = mw == -INFINITY ? 0.f : ex2(mw - M);
        Ls = fmaf(wl[w * MAX_G + n], f, Ls);
        O = fmaf(wo[(w * MAX_G + n) * D + ch], f, O);
      }
    }
    float* rec = a.part + ((size_t)slot * G + n) * PART_STRIDE;
    if (ch == 0) {
      rec[0] = M;
      rec[1] = Ls;
    }
    rec[PART_O + ch] = O;
  }
  tw_sync();  // the window scratch is free again
}

// History items of the token warps.
template <int NG, int GM>
__device__ __forceinline__ void token_warps(const DecodeArgs& a, const Ctx& X, const long long* pre, long long lo,
                                            long long hi, int cta, uint32_t tmem) {
  const CacheView& cv = a.cv;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = threadIdx.x;  // tile row = TMEM lane
  const int G = cv.G, nq = X.nq, GN = G * NG;
  const uint32_t lane_base = (uint32_t)(32 * warp) << 16;
  uint64_t* bars = X.bars;
  const int pg = r >> 6, tok = r & 63;
  // this row's column of the P·s operand (the V^T product's K index) and
  // the power of two of its code position
  const int tT = (tok >> 1) & 3, tI = 2 * (tok >> 4) + ((tok >> 3) & 1), tE = tok & 1;
  const int kidx = 2 * (32 * pg + 8 * tT + tI) + tE;
  const float vfac = (float)(1 << 7) / (float)(1 << code_exp_rt(tI));  // 2^(7 - E)
  float* kc_tab = (float*)(X.smem + X.L.off_kc);
  float* stats = (float*)(X.smem + X.L.off_stats);
  float* red = (float*)(X.smem + X.L.off_red);
  constexpr int KC = MAX_G + MAX_G * 4;
  constexpr int ST = 2 * MAX_G + MAX_G * 4;
  constexpr int NQ = GM * NG <= 16 ? 16 : 32;

  // zero both P·s operands once: rows G·NG .. nq - 1 stay zero
  for (int e = r; e < 2 * X.L.bop_bytes / 16; e += 128)
    ((uint4*)(X.smem + X.L.off_bsv))[e] = make_uint4(0u, 0u, 0u, 0u);

  int g = 0;  // global tile counter
  bool alive = true;
  for_hist_items(cv, a.B, pre, lo, hi, a.bal_wch, cta, [&](const Item& it, int ii) {
    if (!alive) return;
    const int ob = ii & 1;
    // ---- the item's q' operand and logit constants (from the packed query records)
    {
      uint8_t* bq = X.smem + X.L.off_bq + ob * X.L.bop_bytes;
      const int k = r;  // K index of this thread
      const int j = k >> 1, E = k & 1, wi = j >> 3, I = j & 7;
      const int c = 64 * (wi & 1) + 16 * (I >> 1) + 8 * (I & 1) + 2 * (wi >> 1) + E;
      const int gr = c / cv.g;
      const uint8_t* recs = a.qpack + ((size_t)it.b * cv.Hq + it.kvh * G) * QPACK_BYTES;
      for (int n = 0; n < nq; ++n) {
        const int h = n / NG, gg = n % NG;
        __half v = __float2half_rn(0.f);
        if (h < G && gg == gr) v = ((const __half*)(recs + (size_t)h * QPACK_BYTES))[c];
        *(__half*)(bq + bop_offset(nq, n, k)) = v;
      }
      float* kc = kc_tab + ob * KC;
      if (r < G) {
        const uint8_t* rec = recs + (size_t)r * QPACK_BYTES;
        kc[r] = *(const float*)(rec + QPACK_ALPHA) * 16777216.f;  // 2^24: subnormal codes
#pragma unroll
        for (int gr2 = 0; gr2 < NG; ++gr2) {
          float ps = 0.f;
#pragma unroll
          for (int q4 = gr2 * (4 / NG); q4 < (gr2 + 1) * (4 / NG); ++q4) ps += ((const float*)(rec + QPACK_PSUM))[q4];
          kc[MAX_G + r * 4 + gr2] = ps * LOG2E * INV_SQRT_D;
        }
      }
      fence_proxy_async();  // q' is read by the tensor cores (async proxy)
      tw_sync();            // the constants are visible to every token warp
    }
    const float* kc = kc_tab + ob * KC;
    float m_ref[GM], l[GM], zs[GM][NG];
#pragma unroll
    for (int h = 0; h < GM; ++h) {
      m_ref[h] = -INFINITY;
      l[h] = 0.f;
#pragma unroll
      for (int q = 0; q < NG; ++q) zs[h][q] = 0.f;
    }
    const int ntile = (it.p1 - it.p0 + 1) / 2;
    // per-row state kept from a tile's unpack to its softmax
    __half2 ksz_prev[NG], vsz_prev[NG];
    bool valid_prev = false;
    const int hist_b = cv.hist_lens[it.b];
    const int pages_b = (hist_b + PAGE - 1) / PAGE;

    auto softmax = [&](int gt, int t_in_item, const __half2* ksz, const __half2* vsz, bool valid) {
      // S of tile gt: this row's G x NG logit columns
      bool ok = wait_bar(&bars[B_D_FULL + (gt & 1)], (gt >> 1) & 1, X.abort_flag, X.err);
      ok = __all_sync(0xffffffffu, ok);
      float lam[GM];
      if (ok) {
        fence_after();
        uint32_t d[NQ];
        const uint32_t ta = tmem + lane_base + D_COL + nq * (gt & 1);
        if constexpr (NQ == 16) {
          tmem_ld16(ta, d);
          tmem_ld_wait16(d);
        } else {
          tmem_ld32(ta, d);
          tmem_ld_wait32(d);
        }
        fence_before();
        __syncwarp();
        if (lane == 0) arrive(&bars[B_D_EMPTY + (gt & 1)]);
        float2 kz[NG];
#pragma unroll
        for (int q = 0; q < NG; ++q) kz[q] = __half22float2(ksz[q]);
#pragma unroll
        for (int h = 0; h < GM; ++h) {
          float v = 0.f;
          if (h < G) {
#pragma unroll
            for (int q = 0; q < NG; ++q)
              v = fmaf(kz[q].x * kc[h], __uint_as_float(d[h * NG + q]), fmaf(kz[q].y, kc[MAX_G + h * 4 + q], v));
          }
          lam[h] = valid ? v : -INFINITY;
        }
      }
      bool exceed = false;
#pragma unroll
      for (int h = 0; h < GM; ++h) exceed |= (h < G) && (lam[h] > m_ref[h] + TAU);
      // one vote of the 128 rows: some logit passed its threshold, or a wait failed
      const bool fail = tw_any(!ok);
      if (fail) return false;
      if (tw_any(ok && exceed)) {
        // exact maxima of the tile per head, then rescale the running sums and O
        float* wmx = red;
#pragma unroll
        for (int h = 0; h < GM; ++h) {
          if (h < G) {
            float v = lam[h];
#pragma unroll
            for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
            if (lane == 0) wmx[warp * MAX_G + h] = v;
          }
        }
        tw_sync();
        float f[GM];
#pragma unroll
        for (int h = 0; h < GM; ++h) {
          f[h] = 1.f;
          if (h < G) {
            const float tm = fmaxf(fmaxf(wmx[h], wmx[MAX_G + h]), fmaxf(wmx[2 * MAX_G + h], wmx[3 * MAX_G + h]));
            const float mn = fmaxf(m_ref[h], tm);
            f[h] = (m_ref[h] == -INFINITY) ? 0.f : ex2(m_ref[h] - mn);
            m_ref[h] = mn;
            l[h] *= f[h];
#pragma unroll
            for (int q = 0; q < NG; ++q) zs[h][q] *= f[h];
          }
        }
        tw_sync();  // wmx is read by all before the next tile overwrites it
        if (t_in_item > 0) {
          // O holds earlier tiles of this item: wait until their products are
          // done, then scale this row of O (lane r = channel r) per head
          bool ok2 = wait_bar(&bars[B_SV_DONE + ((gt - 1) & 1)], ((gt - 1) >> 1) & 1, X.abort_flag, X.err);
          ok2 = __all_sync(0xffffffffu, ok2);
          if (ok2) {
            fence_after();
            uint32_t o[NQ];
            const uint32_t ta = tmem + lane_base + D_COL + 2 * nq + nq * ob;
            if constexpr (NQ == 16) {
              tmem_ld16(ta, o);
              tmem_ld_wait16(o);
            } else {
              tmem_ld32(ta, o);
              tmem_ld_wait32(o);
            }
#pragma unroll
            for (int n = 0; n < NQ; ++n) {
              if (n < nq) {
                const int h = n / NG;
                o[n] = __float_as_uint(__uint_as_float(o[n]) * (h < G ? f[h < GM ? h : 0] : 1.f));
              }
            }
            if constexpr (NQ == 16) tmem_st16(ta, o);
            else tmem_st32(ta, o);
            tmem_st_wait();
          }
          if (tw_any(!ok2)) return false;
        }
      }
      // P·s of this row into the operand (rows h·NG + q, column kidx)
      if (gt >= 2) {
        bool ok3 = wait_bar(&bars[B_SV_DONE + (gt & 1)], ((gt >> 1) - 1) & 1, X.abort_flag, X.err);
        if (tw_any(!__all_sync(0xffffffffu, ok3))) return false;
      }
      uint8_t* bs = X.smem + X.L.off_bsv + (gt & 1) * X.L.bop_bytes;
      float2 vz[NG];
#pragma unroll
      for (int q = 0; q < NG; ++q) vz[q] = __half22float2(vsz[q]);
#pragma unroll
      for (int h = 0; h < GM; ++h) {
        if (h < G) {
          const float p = valid ? ex2(lam[h] - m_ref[h]) : 0.f;
          l[h] += p;
#pragma unroll
          for (int q = 0; q < NG; ++q) {
            zs[h][q] = fmaf(p, vz[q].y, zs[h][q]);
            *(__half*)(bs + bop_offset(nq, h * NG + q, kidx)) = __float2half_rn(p * vz[q].x * vfac);
          }
        }
      }
      fence_proxy_async();
      fence_before();
      __syncwarp();
      if (lane == 0) arrive(&bars[B_B_FULL + (gt & 1)]);
      return true;
    };

    for (int t = 0; t < ntile && alive; ++t, ++g) {
      const int s = g % NST;
      bool ok = wait_bar(&bars[B_ST_FULL + s], (g / NST) & 1, X.abort_flag, X.err);
      ok = __all_sync(0xffffffffu, ok);
      const int p = it.p0 + 2 * t + pg;
      const bool present = p < it.p1;
      const int flags = ok ? *(volatile int*)(X.smem + X.L.off_flags + 4 * s) : 0;
      const bool copied = present && ((flags >> pg) & 1);
      const int nv = (p == pages_b - 1) ? hist_b - p * PAGE : PAGE;
      const bool valid = copied && tok < nv;
      __half2 ksz[NG], vsz[NG];
      {
        const uint8_t* blk = X.smem + X.L.off_stage + s * X.L.stage_bytes + pg * cv.head_bytes;
        uint4 w0 = make_uint4(0u, 0u, 0u, 0u), w1 = w0;
        if (copied) {
          w0 = *(const uint4*)(blk + tok * 32);
          w1 = *(const uint4*)(blk + tok * 32 + 16);
        }
#pragma unroll
        for (int q = 0; q < NG; ++q) {
          ksz[q] = copied ? *(const __half2*)(blk + off_k_sz() + (tok * NG + q) * 4) : __floats2half2_rn(0.f, 0.f);
          vsz[q] = copied ? *(const __half2*)(blk + off_v_sz(cv.g) + (tok * NG + q) * 4) : __floats2half2_rn(0.f, 0.f);
        }
        // the stage is no longer needed by this warp
        __syncwarp();
        if (lane == 0) arrive(&bars[B_ST_EMPTY + s]);
        uint32_t v[32];
        word_codes(w0.x, v);
        word_codes(w0.y, v + 8);
        word_codes(w0.z, v + 16);
        word_codes(w0.w, v + 24);
        const uint32_t ta = tmem + lane_base + AK_COL + 64 * (g & 1);
        tmem_st32(ta, v);
        word_codes(w1.x, v);
        word_codes(w1.y, v + 8);
        word_codes(w1.z, v + 16);
        word_codes(w1.w, v + 24);
        tmem_st32(ta + 32, v);
        tmem_st_wait();
        fence_before();
        __syncwarp();
        if (lane == 0) arrive(&bars[B_AK_FULL + (g & 1)]);
      }
      if (tw_any(!ok)) {
        alive = false;
        break;
      }
      if (t > 0 && !softmax(g - 1, t - 1, ksz_prev, vsz_prev, valid_prev)) {
        alive = false;
        break;
      }
#pragma unroll
      for (int q = 0; q < NG; ++q) {
        ksz_prev[q] = ksz[q];
        vsz_prev[q] = vsz[q];
      }
      valid_prev = valid;
    }
    if (alive && ntile > 0 && !softmax(g - 1, ntile - 1, ksz_prev, vsz_prev, valid_prev)) alive = false;
    if (!alive) return;
    // ---- the item's sums: l and zs over the 128 rows -> stats of parity ob
    if (ii >= 2) {
      bool ok = wait_bar(&bars[B_O_EMPTY + ob], ((ii >> 1) - 1) & 1, X.abort_flag, X.err);
      if (tw_any(!__all_sync(0xffffffffu, ok))) {
        alive = false;
        return;
      }
    }
#pragma unroll
    for (int h = 0; h < GM; ++h) {
      if (h < G) {
        float v = l[h];
#pragma unroll
        for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == 0) red[warp * KC + h] = v;
#pragma unroll
        for (int q = 0; q < NG; ++q) {
          float z = zs[h][q];
#pragma unroll
          for (int o = 16; o; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
          if (lane == 0) red[warp * KC + MAX_G + h * 4 + q] = z;
        }
      }
    }
    tw_sync();
    float* st = stats + ob * ST;
    if (r == 0) {
#pragma unroll
      for (int h = 0; h < GM; ++h)
        if (h < G) st[h] = m_ref[h];  // the same in every row
    }
    if (r < G) st[MAX_G + r] = red[r] + red[KC + r] + red[2 * KC + r] + red[3 * KC + r];
    if (r < GN) {
      const int h = r / NG, q = r % NG, e = MAX_G + h * 4 + q;
      st[2 * MAX_G + h * 4 + q] = red[e] + red[KC + e] + red[2 * KC + e] + red[3 * KC + e];
    }
    tw_sync();
    if (lane == 0) arrive(&bars[B_STATS + ob]);
  });
}

// ---------------------------------------------------------- channel warps
template <int NG, int GM>
__device__ __forceinline__ void channel_warps(const DecodeArgs& a, const Ctx& X, const long long* pre, long long lo,
                                              long long hi, int cta, uint32_t tmem) {
  const CacheView& cv = a.cv;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ch = threadIdx.x - 32 * CW;  // rotated channel = TMEM lane
  const int G = cv.G, nq = X.nq;
  const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
  uint64_t* bars = X.bars;
  const float* stats = (const float*)(X.smem + X.L.off_stats);
  constexpr int ST = 2 * MAX_G + MAX_G * 4;
  constexpr int NQ = GM * NG <= 16 ? 16 : 32;
  const int gr = ch / cv.g;
  int g = 0;
  bool alive = true;
  for_hist_items(cv, a.B, pre, lo, hi, a.bal_wch, cta, [&](const Item& it, int ii) {
    if (!alive) return;
    const int ob = ii & 1;
    const int ntile = (it.p1 - it.p0 + 1) / 2;
    for (int t = 0; t < ntile; ++t, ++g) {
      const int s = g % NST;
      bool ok = wait_bar(&bars[B_ST_FULL + s], (g / NST) & 1, X.abort_flag, X.err);
      if (ok && g >= 2) ok = wait_bar(&bars[B_SV_DONE + (g & 1)], ((g >> 1) - 1) & 1, X.abort_flag, X.err);
      if (!__all_sync(0xffffffffu, ok)) {
        alive = false;
        return;
      }
      const int flags = *(volatile int*)(X.smem + X.L.off_flags + 4 * s);
      const uint8_t* st = X.smem + X.L.off_stage + s * X.L.stage_bytes;
      uint4 w0 = make_uint4(0u, 0u, 0u, 0u), w1 = w0;
      if (flags & 1) w0 = *(const uint4*)(st + 2048 + ch * 16);
      if (flags & 2) w1 = *(const uint4*)(st + cv.head_bytes + 2048 + ch * 16);
      __syncwarp();
      if (lane == 0) arrive(&bars[B_ST_EMPTY + s]);
      // column 32 pg + 8 T + I = code pair I of word T of page pg
      uint32_t v[32];
      word_codes(w0.x, v);
      word_codes(w0.y, v + 8);
      word_codes(w0.z, v + 16);
      word_codes(w0.w, v + 24);
      const uint32_t ta = tmem + lane_base + AV_COL + 64 * (g & 1);
      tmem_st32(ta, v);
      word_codes(w1.x, v);
      word_codes(w1.y, v + 8);
      word_codes(w1.z, v + 16);
      word_codes(w1.w, v + 24);
      tmem_st32(ta + 32, v);
      tmem_st_wait();
      fence_before();
      __syncwarp();
      if (lane == 0) arrive(&bars[B_AV_FULL + (g & 1)]);
    }
    // ---- the item's output: O (this channel's row) and the token warps' sums
    bool ok = wait_bar(&bars[B_O_FULL + ob], (ii >> 1) & 1, X.abort_flag, X.err);
    if (ok) ok = wait_bar(&bars[B_STATS + ob], (ii >> 1) & 1, X.abort_flag, X.err);
    if (!__all_sync(0xffffffffu, ok)) {
      alive = false;
      return;
    }
    fence_after();
    uint32_t o[NQ];
    const uint32_t ta = tmem + lane_base + D_COL + 2 * nq + nq * ob;
    if constexpr (NQ == 16) {
      tmem_ld16(ta, o);
      tmem_ld_wait16(o);
    } else {
      tmem_ld32(ta, o);
      tmem_ld_wait32(o);
    }
    const float* sm = stats + ob * ST;
#pragma unroll
    for (int h = 0; h < GM; ++h) {
      if (h < G) {
        // this channel's group column of head h
        float ov = 0.f;
#pragma unroll
        for (int q = 0; q < NG; ++q) ov = (q == gr) ? __uint_as_float(o[h * NG + q]) : ov;
        // o' = 2^17 * O + sum p z  (P·s carried 2^(7 - E), the codes 2^(E - 24))
        const float val = fmaf(ov, 131072.f, sm[2 * MAX_G + h * 4 + gr]);
        float* rec = a.part + ((size_t)it.slot * G + h) * PART_STRIDE;
        rec[PART_O + ch] = val;
        if (ch == 0) {
          rec[0] = sm[h];
          rec[1] = sm[MAX_G + h];
        }
      }
    }
    fence_before();
    __syncwarp();
    if (lane == 0) arrive(&bars[B_O_EMPTY + ob]);
  });
}

// --------------------------------------------------------------- mma warp
__device__ __forceinline__ void mma_thread(const DecodeArgs& a, const Ctx& X, const long long* pre, long long lo,
                                           long long hi, int cta, uint32_t tmem) {
  uint64_t* bars = X.bars;
  const int nq = X.nq;
  const uint32_t id = idesc(nq);
  int g = 0;
  bool alive = true;
  auto sv = [&](int gt, int t_in_item, int ii) -> bool {
    const int ob = ii & 1;
    if (!wait_bar(&bars[B_B_FULL + (gt & 1)], (gt >> 1) & 1, X.abort_flag, X.err)) return false;
    if (!wait_bar(&bars[B_AV_FULL + (gt & 1)], (gt >> 1) & 1, X.abort_flag, X.err)) return false;
    if (t_in_item == 0 && ii >= 2 && !wait_bar(&bars[B_O_EMPTY + ob], ((ii >> 1) - 1) & 1, X.abort_flag, X.err))
      return false;
    fence_after();
    const uint32_t bsv = X.sbase + X.L.off_bsv + (gt & 1) * X.L.bop_bytes;
    const uint32_t d = tmem + D_COL + 2 * nq + nq * ob;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk)
      mma_ts(d, tmem + AV_COL + 64 * (gt & 1) + 8 * kk, sdesc(bsv + (kk >> 2) * (nq * 128) + (kk & 3) * 32), id,
             (t_in_item > 0 || kk > 0) ? 1u : 0u);
    commit(&bars[B_SV_DONE + (gt & 1)]);
    return true;
  };
  for_hist_items(a.cv, a.B, pre, lo, hi, a.bal_wch, cta, [&](const Item& it, int ii) {
    if (!alive) return;
    const int ntile = (it.p1 - it.p0 + 1) / 2;
    const uint32_t bq = X.sbase + X.L.off_bq + (ii & 1) * X.L.bop_bytes;
    for (int t = 0; t < ntile; ++t, ++g) {
      if (!wait_bar(&bars[B_AK_FULL + (g & 1)], (g >> 1) & 1, X.abort_flag, X.err) ||
          (g >= 2 && !wait_bar(&bars[B_D_EMPTY + (g & 1)], ((g >> 1) - 1) & 1, X.abort_flag, X.err))) {
        alive = false;
        return;
      }
      fence_after();
      const uint32_t d = tmem + D_COL + nq * (g & 1);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks)
        mma_ts(d, tmem + AK_COL + 64 * (g & 1) + 8 * ks, sdesc(bq + (ks >> 2) * (nq * 128) + (ks & 3) * 32), id,
               ks > 0 ? 1u : 0u);
      commit(&bars[B_D_FULL + (g & 1)]);
      if (t > 0 && !sv(g - 1, t - 1, ii)) {
        alive = false;
        return;
      }
    }
    if (ntile > 0) {
      if (!sv(g - 1, ntile - 1, ii)) {
        alive = false;
        return;
      }
      commit(&bars[B_O_FULL + (ii & 1)]);
    }
  });
  // every issued product completes before the tensor memory is released
  commit(&bars[B_DRAIN]);
  mbar_wait(&bars[B_DRAIN], 0);
}

// ------------------------------------------------------------- page copies
__device__ __forceinline__ void loader_warp(const DecodeArgs& a, const Ctx& X, const long long* pre, long long lo,
                                            long long hi, int cta) {
  const CacheView& cv = a.cv;
  const int lane = threadIdx.x & 31;
  uint64_t* bars = X.bars;
  const int hb = cv.head_bytes;
  int g = 0, issued = 0;
  bool alive = true;
  for_hist_items(cv, a.B, pre, lo, hi, a.bal_wch, cta, [&](const Item& it, int) {
    if (!alive) return;
    const int32_t* ptab = cv.page_table + (size_t)it.b * cv.max_pages_per_req;
    const int np = it.p1 - it.p0;
    for (int base = 0; base < np && alive; base += 32) {
      const int mine = base + lane < np ? __ldg(ptab + it.p0 + base + lane) : -1;
      const int cnt = np - base < 32 ? np - base : 32;
      for (int j = 0; j < cnt; j += 2, ++g) {
        const int pa = __shfl_sync(0xffffffffu, mine, j);
        const int pb = __shfl_sync(0xffffffffu, mine, (j + 1) & 31);
        const bool has_b = j + 1 < cnt;
        int go = 1;
        if (lane == 0) {
          const int s = g % NST;
          if (g >= NST && !wait_bar(&bars[B_ST_EMPTY + s], ((g / NST) - 1) & 1, X.abort_flag, X.err)) {
            go = 0;
          } else {
            const bool oka = pa >= 0 && pa < cv.num_pages;
            const bool okb = has_b && pb >= 0 && pb < cv.num_pages;
            if (!oka) record_error(cv.err, pa < 0 ? OSCAR_ERR_NO_PAGE : OSCAR_ERR_RANGE);
            if (has_b && !okb) record_error(cv.err, pb < 0 ? OSCAR_ERR_NO_PAGE : OSCAR_ERR_RANGE);
            *(volatile int*)(X.smem + X.L.off_flags + 4 * s) = (oka ? 1 : 0) | (okb ? 2 : 0);
            uint8_t* dst = X.smem + X.L.off_stage + s * X.L.stage_bytes;
            mbar_expect_tx(&bars[B_ST_FULL + s], (uint32_t)hb * ((oka ? 1u : 0u) + (okb ? 1u : 0u)));
            if (oka)
              bulk_g2s(dst, cv.pool + (size_t)pa * cv.page_bytes + (size_t)it.kvh * hb, (uint32_t)hb,
                       &bars[B_ST_FULL + s]);
            if (okb)
              bulk_g2s(dst + hb, cv.pool + (size_t)pb * cv.page_bytes + (size_t)it.kvh * hb, (uint32_t)hb,
                       &bars[B_ST_FULL + s]);
            issued = g + 1;
          }
        }
        go = __shfl_sync(0xffffffffu, go, 0);
        if (!go) {
          alive = false;
          break;
        }
      }
    }
  });
  // every copy this CTA started has landed before it exits
  if (lane == 0)
    for (int i = issued - NST < 0 ? 0 : issued - NST; i < issued; ++i) mbar_wait(&bars[B_ST_FULL + i % NST], (i / NST) & 1);
}

// ------------------------------------------------------------------ kernel
template <int NG, int GM>
__global__ void __launch_bounds__(THREADS, 1) decode_tc_kernel(DecodeArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - ((uint32_t)__cvta_generic_to_shared(smem_raw) & 1023)) & 1023);
  const CacheView& cv = a.cv;
  const int tid = threadIdx.x, warp = tid >> 5;
  Ctx X;
  X.smem = smem;
  X.sbase = (uint32_t)__cvta_generic_to_shared(smem);
  X.L = layout(cv.head_bytes, a.B);
  X.bars = (uint64_t*)(smem + X.L.off_bar);
  int* misc = (int*)(smem + X.L.off_misc);
  X.abort_flag = misc + 1;
  X.err = cv.err;
  X.nq = GM * NG <= 16 ? 16 : 32;
  long long* pre = (long long*)(smem + X.L.off_pre);

  pdl_launch_dependents();  // merge_kernel may be scheduled as CTAs of this grid retire
  if (tid == 0) {
    for (int i = 0; i < NST; ++i) {
      mbar_init(&X.bars[B_ST_FULL + i], 1);
      mbar_init(&X.bars[B_ST_EMPTY + i], 8);  // four token warps and four channel warps
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&X.bars[B_AK_FULL + i], 4);
      mbar_init(&X.bars[B_AV_FULL + i], 4);
      mbar_init(&X.bars[B_D_FULL + i], 1);
      mbar_init(&X.bars[B_D_EMPTY + i], 4);
      mbar_init(&X.bars[B_B_FULL + i], 4);
      mbar_init(&X.bars[B_SV_DONE + i], 1);
      mbar_init(&X.bars[B_O_FULL + i], 1);
      mbar_init(&X.bars[B_O_EMPTY + i], 4);
      mbar_init(&X.bars[B_STATS + i], 4);
    }
    mbar_init(&X.bars[B_DRAIN], 1);
    misc[1] = 0;
  }
  if (warp == MMA_WARP) {  // whole warp: allocate the tensor memory, publish its address
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(
                     (uint32_t)__cvta_generic_to_shared(&misc[0])),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
  }
  fence_proxy_async();
  // the lengths and page tables come from earlier stream work: readable before the wait
  const Balanced bl = make_balanced(cv.seq_lens, cv.hist_lens, a.B, cv.Hkv, a.bal_wch, gridDim.x, pre);
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = (uint32_t)misc[0];
  const int cta = blockIdx.x;
  const bool part_of = cta < bl.n;
  const long long lo = part_of ? balanced_lo(bl, cta) : 0, hi = part_of ? balanced_lo(bl, cta + 1) : 0;

  if (warp < CW) {
    pdl_wait();  // q' (prep) and the window contents (append) are ready from here on
    // ---- the BF16 window chunks whose first position lies in this CTA's range
    for_segments(cv, a.B, pre, lo, hi, a.bal_wch, [&](int b, int kvh, long long seg, int P, unsigned mask) {
      long long x = seg + P;
      for (int c = 0; c < WIN_CHUNKS; ++c) {
        if (!((mask >> c) & 1u)) continue;
        if (x >= lo && x < hi)
          tw_window_chunk(a, X, b, kvh, c, bl.n + a.B * cv.Hkv + WIN_CHUNKS * (b * cv.Hkv + kvh) + c);
        x += a.bal_wch;
      }
    });
    token_warps<NG, GM>(a, X, pre, lo, hi, cta, tmem);
  } else if (warp < LD_WARP) {
    channel_warps<NG, GM>(a, X, pre, lo, hi, cta, tmem);
  } else if (warp == LD_WARP) {
    loader_warp(a, X, pre, lo, hi, cta);
  } else if ((tid & 31) == 0) {
    mma_thread(a, X, pre, lo, hi, cta, tmem);
  }
  if (warp >= CW) pdl_wait();  // every warp has waited before the grid ends
  fence_before();
  __syncthreads();
  fence_after();
  if (warp == MMA_WARP)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(tmem), "r"(TMEM_COLS) : "memory");
}

template <int NG, int GM>
cudaError_t launch_tc_t(const DecodeArgs& a, cudaStream_t st) {
  const Layout L = layout(a.cv.head_bytes, a.B);
  static int limit[MAX_DEVICES];
  const cudaError_t e = raise_smem_limit(decode_tc_kernel<NG, GM>, limit, L.total);
  if (e != cudaSuccess) return e;
  return launch_pdl(decode_tc_kernel<NG, GM>, dim3(a.bal_grid), dim3(THREADS), L.total, st, a);
}

}  // namespace

int decode_tc_smem_bytes(int head_bytes, int B) { return layout(head_bytes, B).total; }
int decode_tc_window_weight() { return WCH; }

cudaError_t launch_decode_tc(const DecodeArgs& a, cudaStream_t st) {
  if (a.cv.G <= 4) {
    if (a.cv.NG == 1) return launch_tc_t<1, 4>(a, st);
    if (a.cv.NG == 2) return launch_tc_t<2, 4>(a, st);
    return launch_tc_t<4, 4>(a, st);
  }
  if (a.cv.NG == 1) return launch_tc_t<1, 8>(a, st);
  if (a.cv.NG == 2) return launch_tc_t<2, 8>(a, st);
  return launch_tc_t<4, 8>(a, st);
}

}  // namespace oscar
