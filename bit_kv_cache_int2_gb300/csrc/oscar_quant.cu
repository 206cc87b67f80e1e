// Demotion, bulk import and quantiser test hooks of liboscar (sm_103a).
//
// The demotion step follows the pipeline figure of "超越TurboQuant：Together AI把
// 2-bit KV Cache推向真实服务" ("从离线校准到在线推理的pipeline" and the paragraph
// under it): a new token is written to the BF16 recent window, and the oldest
// recent token is rotated, clipped, quantised and packed 4 codes per byte into
// INT2 history.  Region sizes (sink 64, recent 256) are from "Together AI 开源
// OSCAR：一种面向长上下文 LLM 服务的注意力感知 2 位 KV 缓存量化系统", section
// "服务系统：混合精度缓存布局".
#include "oscar_internal.cuh"

namespace oscar {

namespace {

// Quantise the rotated value y (channel j of a 128-thread group) and place its
// code in a K row (kw: 8 words of smem, zeroed) or in a V block word in smem
// (vblk: 512 words, channel-major, zeroed) for token row t.  Writes (s, z)
// through sz_out (token row t of an [64][NG] half2 array) for the group leader.
__device__ __forceinline__ void quant_pack(float y, int j, int g, float clip, QThr th, float* red, int bar,
                                           bool is_v, int t, uint32_t* kw, uint32_t* vblk,
                                           __half2* sz_row) {
  float mn, mx;
  group_minmax(y, j, g, red, bar, mn, mx);
  const QParams qp = quant_params(mn, mx, clip);
  const uint32_t code = quant_code(y, qp, th);
  if (!is_v) {
    atomicOr(&kw[k_word(j)], code << k_bit(j));
  } else {
    atomicOr(&vblk[j * 4 + v_word(t)], code << v_bit(t));
  }
  if ((j % g) == 0) sz_row[j / g] = __halves2half2(qp.s, qp.z);
}

// Same, but writing a single token's V code straight into a V block in global
// memory: its two bits of the owning word are cleared and set by two atomic
// reductions (one writer per word; same-address atomics of a thread keep their
// order), so no load of the word sits on the demotion's critical path.
__device__ __forceinline__ void quant_store_v_global(float y, int j, int g, float clip, QThr th, float* red,
                                                     int bar, int t, uint32_t* vblk_g,
                                                     __half2* sz_row) {
  float mn, mx;
  group_minmax(y, j, g, red, bar, mn, mx);
  const QParams qp = quant_params(mn, mx, clip);
  const uint32_t code = quant_code(y, qp, th);
  uint32_t* wp = vblk_g + j * 4 + v_word(t);
  const uint32_t sh = (uint32_t)v_bit(t);
  atomicAnd(wp, ~(3u << sh));
  atomicOr(wp, code << sh);
  if ((j % g) == 0) sz_row[j / g] = __halves2half2(qp.s, qp.z);
}

// ------------------------------------------------------------------ append
// grid = (B * Hkv, 2): blockIdx.y = 0 handles K, 1 handles V.  block = 512:
// four parts of 128 threads split the 128-row matvec x·R so that all of R's
// loads are in flight at once; threads 0..127 then finish the token.
// One (request, kv head, K|V) of the append, by 512 threads; bk = request *
// Hkv + kv head, isv = 0 for K, 1 for V.  The body waits for earlier stream
// work after issuing its rotation-table loads; with `release` it then lets
// its dependents launch at once, otherwise the caller releases them later.
// With `pred` (a decode step) the K CTA of kv head 0 first writes the lengths
// this append will leave, pred[b] (sequence), pred[B + b] (history) and
// pred[2B + b] (history before), and every CTA releases its dependents once
// that is done and fenced.
__device__ __forceinline__ void append_body(const CacheView& cv, const LayerRot& rot,
                                            const __nv_bfloat16* __restrict__ knew,
                                            const __nv_bfloat16* __restrict__ vnew, int do_append,
                                            int* req_counter, int bk, int isv, bool release,
                                            int32_t* pred = nullptr, int B = 0) {
  __shared__ float xs[D];
  __shared__ float part[4][D];
  __shared__ float red[8];
  __shared__ uint32_t kw[8];
  __shared__ int st[6];
  const int b = bk / cv.Hkv, h = bk % cv.Hkv;
  const int t = threadIdx.x, j = t & 127, pp = t >> 7;
  // R's loads do not depend on earlier stream work: start them first
  float u[32];
  {
    const float* R = (isv ? rot.R_V : rot.R_K) + (size_t)h * D * D + (size_t)(32 * pp) * D + j;
#pragma unroll
    for (int k = 0; k < 32; ++k) u[k] = __ldg(R + k * D);
  }
  // The lengths, the page-table entry and the ring slot are dependent round
  // trips after the wait: bring their lines into L2 now (hints only; the
  // values are read after the wait).  Thread t takes line t of this head's
  // 64 KB ring block; the request's page-table row is spread over its 2 Hkv CTAs.
  {
    const __nv_bfloat16* rb = (isv ? cv.ring_v : cv.ring_k) + (size_t)(b * cv.Hkv + h) * RECENT * D;
    if (t < RECENT * D * 2 / 128) asm volatile("prefetch.global.L2 [%0];\n" ::"l"((const char*)rb + 128 * t));
    if (t == 0) asm volatile("prefetch.global.L2 [%0];\n" ::"l"(cv.hist_lens + b));
    const int per_req = 2 * cv.Hkv, me = 2 * h + isv;
    const int lines = (cv.max_pages_per_req + 31) / 32;
    for (int l = me + per_req * t; l < lines; l += per_req * (int)blockDim.x)
      asm volatile("prefetch.global.L2 [%0];\n" ::"l"(cv.page_table + (size_t)b * cv.max_pages_per_req + 32 * (size_t)l));
  }
  // the new tokens, the lengths and the cache belong to earlier stream work;
  // the decode's prep_kernel waits for this grid before it reads anything
  pdl_wait();
  if (release && !pred) pdl_launch_dependents();
  if (t == 0) {
    const int L = cv.seq_lens[b], H = cv.hist_lens[b];
    const int recent = L > SINK ? L - SINK - H : 0;
    int ok = (L >= 0 && H >= 0 && H <= (L > SINK ? L - SINK : 0) && recent <= RECENT);
    if (!ok) record_error(cv.err, OSCAR_ERR_STATE);
    const int demote = ok && (do_append ? (recent == RECENT) : (recent > 0));
    int page = -1;
    if (demote) {
      const int pi = H / PAGE;
      if (pi >= cv.max_pages_per_req) {
        ok = 0;
        record_error(cv.err, OSCAR_ERR_RANGE);
      } else {
        page = cv.page_table[(size_t)b * cv.max_pages_per_req + pi];
        if (page < 0) {
          ok = 0;
          record_error(cv.err, OSCAR_ERR_NO_PAGE);
        } else if (page >= cv.num_pages) {
          ok = 0;
          record_error(cv.err, OSCAR_ERR_RANGE);
        }
      }
    }
    st[0] = L;
    st[1] = H;
    st[2] = ok && demote;
    st[3] = page;
    st[4] = ok;
    if (pred && h == 0 && !isv) {
      // the lengths the last CTA of the request writes below
      pred[b] = ok ? L + do_append : L;
      pred[B + b] = ok ? H + (demote ? 1 : 0) : H;
      pred[2 * B + b] = H;
      __threadfence();
    }
  }
  if (t < 8) kw[t] = 0u;
  __syncthreads();
  if (release && pred) pdl_launch_dependents();
  const int L = st[0], H = st[1], demote = st[2], page = st[3], ok = st[4];
  const size_t head = (size_t)(b * cv.Hkv + h);
  __nv_bfloat16* ring = isv ? cv.ring_v : cv.ring_k;

  if (demote) {
    const int ring_slot = H % RECENT;  // absolute position 64 + H
    if (t < D) xs[t] = __bfloat162float(ring[(head * RECENT + ring_slot) * D + t]);
    __syncthreads();
    float acc = 0.f;
#pragma unroll
    for (int k = 0; k < 32; ++k) acc = fmaf(xs[32 * pp + k], u[k], acc);
    part[pp][j] = acc;
    __syncthreads();
    if (pp == 0) {
      const float y = (part[0][j] + part[1][j]) + (part[2][j] + part[3][j]);
      const float clip = (isv ? rot.clip_v : rot.clip_k)[h];
      const QThr th = quant_thr(rot.cb + (size_t)(isv * cv.Hkv + h) * CB_WORDS);
      uint8_t* blk = cv.pool + (size_t)page * cv.page_bytes + (size_t)h * cv.head_bytes;
      const int tr = H % PAGE;
      if (!isv) {
        quant_pack(y, j, cv.g, clip, th, red, 1, false, tr, kw, nullptr,
                   (__half2*)(blk + off_k_sz()) + tr * cv.NG);
        group_sync(1);
        if (t < 8) ((uint32_t*)(blk + tr * 32))[t] = kw[t];
      } else {
        quant_store_v_global(y, j, cv.g, clip, th, red, 1, tr, (uint32_t*)(blk + 2048),
                             (__half2*)(blk + off_v_sz(cv.g)) + tr * cv.NG);
      }
    }
  }
  __syncthreads();  // the evicted ring slot is fully read before it is overwritten

  if (do_append && ok && t < 16) {
    const __nv_bfloat16* src = (isv ? vnew : knew) + head * D;
    __nv_bfloat16* dst;
    if (L < SINK)
      dst = (isv ? cv.sink_v : cv.sink_k) + (head * SINK + L) * D;
    else
      dst = ring + (head * RECENT + (L - SINK) % RECENT) * D;
    ((uint4*)dst)[t] = ((const uint4*)src)[t];
  }
  // The last CTA of request b to finish updates its lengths: every CTA of the
  // request has read the old lengths before it increments the counter.  In a
  // decode step (pred) the merge kernel writes them instead, from pred.
  __syncthreads();
  if (t == 0 && !pred) {
    // release: this CTA's reads of the old lengths come before the count;
    // acquire: the last CTA writes the lengths after every CTA's reads
    const int old = atomic_add_acq_rel_gpu(&req_counter[b], 1);
    if (old == 2 * cv.Hkv - 1) {
      req_counter[b] = 0;
      if (ok) {
        cv.seq_lens[b] = L + (do_append ? 1 : 0);
        cv.hist_lens[b] = H + demote;
      }
    }
  }
}


// grid = (B * Hkv, 2): blockIdx.y = 0 handles K, 1 handles V.
__global__ void __launch_bounds__(512) append_kernel(CacheView cv, LayerRot rot,
                                                     const __nv_bfloat16* __restrict__ knew,
                                                     const __nv_bfloat16* __restrict__ vnew,
                                                     int do_append, int* req_counter) {
  append_body(cv, rot, knew, vnew, do_append, req_counter, blockIdx.x, blockIdx.y, true);
}

// One decode step's first kernel, grid = (B * Hkv, 3), block 512: y = 0 / 1
// append K / V of (request, kv head) x (as append_kernel), y = 2 computes the
// packed query of x, its four 128-thread parts taking one channel quarter
// each (as prep_kernel).  The query rotation does not depend on the append,
// so the two run side by side.
// With a.step_pred (the mma.sync decode kernels) every CTA releases the
// decode kernel right after its wait, the K CTAs of kv head 0 once they have
// published the lengths the append will leave; the decode kernel schedules
// from those, copies the history pages the append does not write, and waits
// for this grid before it reads anything else.  Otherwise (the tensor-memory
// kernel reads the cache state before its wait) each CTA releases only once
// its own writes are done and fenced.
__global__ void __launch_bounds__(512) step_kernel(CacheView cv, LayerRot rot,
                                                   const __nv_bfloat16* __restrict__ knew,
                                                   const __nv_bfloat16* __restrict__ vnew,
                                                   int* req_counter, DecodeArgs a) {
  __shared__ PrepSmem psm[4];
  const int bk = blockIdx.x;
  const bool early = a.step_pred != 0;
  if (blockIdx.y < 2) {
    append_body(cv, rot, knew, vnew, 1, req_counter, bk, blockIdx.y, early, early ? a.pred : nullptr, a.B);
  } else {
    prep_body(a, bk, threadIdx.x >> 7, threadIdx.x & 127, psm[threadIdx.x >> 7], early);
  }
  if (!early) {
    __syncthreads();
    __threadfence();
    pdl_launch_dependents();
  }
}

// ------------------------------------------------------------------ import
// Copies the sink and recent tokens of an n-token prefix; checks emptiness.
// grid = B * Hkv, block = 256.
__global__ void __launch_bounds__(256) import_window_kernel(CacheView cv,
                                                            const __nv_bfloat16* __restrict__ K,
                                                            const __nv_bfloat16* __restrict__ V,
                                                            int n) {
  const int b = blockIdx.x / cv.Hkv, h = blockIdx.x % cv.Hkv;
  if (cv.seq_lens[b] != 0) {
    if (threadIdx.x == 0 && h == 0) record_error(cv.err, OSCAR_ERR_STATE);
    return;
  }
  const size_t head = (size_t)(b * cv.Hkv + h);
  const uint4* srcK = (const uint4*)(K + head * (size_t)n * D);
  const uint4* srcV = (const uint4*)(V + head * (size_t)n * D);
  const int nsink = n < SINK ? n : SINK;
  const int r0 = (n - RECENT) > SINK ? n - RECENT : SINK;  // first recent position
  const int nrec = n > r0 ? n - r0 : 0;
  // 16 uint4 per token row
  for (int idx = threadIdx.x; idx < nsink * 16; idx += blockDim.x) {
    const int p = idx >> 4, c = idx & 15;
    ((uint4*)(cv.sink_k + (head * SINK + p) * D))[c] = srcK[(size_t)p * 16 + c];
    ((uint4*)(cv.sink_v + (head * SINK + p) * D))[c] = srcV[(size_t)p * 16 + c];
  }
  for (int idx = threadIdx.x; idx < nrec * 16; idx += blockDim.x) {
    const int p = r0 + (idx >> 4), c = idx & 15;
    const int slot = (p - SINK) % RECENT;
    ((uint4*)(cv.ring_k + (head * RECENT + slot) * D))[c] = srcK[(size_t)p * 16 + c];
    ((uint4*)(cv.ring_v + (head * RECENT + slot) * D))[c] = srcV[(size_t)p * 16 + c];
  }
}

__device__ __forceinline__ uint8_t* lookup_page(const CacheView& cv, int b, int pi, bool report) {
  if (pi >= cv.max_pages_per_req) {
    if (report) record_error(cv.err, OSCAR_ERR_RANGE);
    return nullptr;
  }
  const int page = cv.page_table[(size_t)b * cv.max_pages_per_req + pi];
  if (page < 0) {
    if (report) record_error(cv.err, OSCAR_ERR_NO_PAGE);
    return nullptr;
  }
  if (page >= cv.num_pages) {
    if (report) record_error(cv.err, OSCAR_ERR_RANGE);
    return nullptr;
  }
  return cv.pool + (size_t)page * cv.page_bytes;
}

constexpr int IMP_NT = 8;  // tokens rotated together (one U load feeds 8 FMAs)

// Quantises one history page of one kv head: grid (B * Hkv, pages), block 256.
__global__ void __launch_bounds__(256) import_int2_pages_kernel(CacheView cv, LayerRot rot,
                                                                const __nv_bfloat16* __restrict__ K,
                                                                const __nv_bfloat16* __restrict__ V,
                                                                int n) {
  __shared__ float xs[2][IMP_NT][D];
  __shared__ float red[2][8];
  __shared__ __align__(16) uint32_t kwords[PAGE * 8];
  __shared__ __align__(16) uint32_t vwords[D * 4];
  __shared__ __align__(16) __half2 szs[2][PAGE * 4];
  const int b = blockIdx.x / cv.Hkv, h = blockIdx.x % cv.Hkv, pg = blockIdx.y;
  const int hist = n > SINK + RECENT ? n - SINK - RECENT : 0;
  const int t0 = pg * PAGE;
  if (t0 >= hist) return;
  if (cv.seq_lens[b] != 0) return;  // reported by import_window_kernel
  uint8_t* page = lookup_page(cv, b, pg, h == 0 && threadIdx.x == 0);
  if (!page) return;
  uint8_t* blk = page + (size_t)h * cv.head_bytes;
  const int nt = (hist - t0) < PAGE ? hist - t0 : PAGE;
  const int grp = threadIdx.x >> 7, j = threadIdx.x & 127, bar = 1 + grp;
  for (int i = threadIdx.x; i < PAGE * 8; i += 256) kwords[i] = 0u;
  for (int i = threadIdx.x; i < D * 4; i += 256) vwords[i] = 0u;
  for (int i = threadIdx.x; i < 2 * PAGE * 4; i += 256) (&szs[0][0])[i] = __halves2half2(__float2half(0.f), __float2half(0.f));
  const size_t head = (size_t)(b * cv.Hkv + h);
  const __nv_bfloat16* src = (grp == 0 ? K : V) + (head * (size_t)n + SINK + t0) * D;
  const float* R = (grp == 0 ? rot.R_K : rot.R_V) + (size_t)h * D * D;
  const float clip = (grp == 0 ? rot.clip_k : rot.clip_v)[h];
  const QThr th = quant_thr(rot.cb + (size_t)(grp * cv.Hkv + h) * CB_WORDS);
  __syncthreads();
  for (int tb = 0; tb < nt; tb += IMP_NT) {
    const int cnt = (nt - tb) < IMP_NT ? nt - tb : IMP_NT;
    for (int k = 0; k < IMP_NT; ++k)
      xs[grp][k][j] = k < cnt ? __bfloat162float(src[(size_t)(tb + k) * D + j]) : 0.f;
    group_sync(bar);
    float acc[IMP_NT];
#pragma unroll
    for (int k = 0; k < IMP_NT; ++k) acc[k] = 0.f;
    for (int i = 0; i < D; ++i) {
      const float r = __ldg(R + i * D + j);
#pragma unroll
      for (int k = 0; k < IMP_NT; ++k) acc[k] = fmaf(xs[grp][k][i], r, acc[k]);
    }
    for (int k = 0; k < cnt; ++k) {
      const float y = acc[k];
      const int t = tb + k;
      quant_pack(y, j, cv.g, clip, th, red[grp], bar, grp == 1, t, kwords + t * 8, vwords,
                 &szs[grp][t * cv.NG]);
    }
    group_sync(bar);
  }
  __syncthreads();
  // write the block: K codes 2048 B, V codes 2048 B, K s/z, V s/z
  uint4* dst = (uint4*)blk;
  for (int i = threadIdx.x; i < 128; i += 256) dst[i] = ((const uint4*)kwords)[i];
  for (int i = threadIdx.x; i < 128; i += 256) dst[128 + i] = ((const uint4*)vwords)[i];
  const int szq = PAGE * cv.NG * 4 / 16;  // uint4 per s/z array
  for (int i = threadIdx.x; i < szq; i += 256) {
    ((uint4*)(blk + off_k_sz()))[i] = ((const uint4*)szs[0])[i];
    ((uint4*)(blk + off_v_sz(cv.g)))[i] = ((const uint4*)szs[1])[i];
  }
}

// Copies BF16 history tokens into a BF16 page: grid (B * Hkv, pages), block 256.
__global__ void __launch_bounds__(256) import_bf16_pages_kernel(CacheView cv,
                                                                const __nv_bfloat16* __restrict__ K,
                                                                const __nv_bfloat16* __restrict__ V,
                                                                int n) {
  const int b = blockIdx.x / cv.Hkv, h = blockIdx.x % cv.Hkv, pg = blockIdx.y;
  const int hist = n > SINK + RECENT ? n - SINK - RECENT : 0;
  const int t0 = pg * PAGE;
  if (t0 >= hist) return;
  if (cv.seq_lens[b] != 0) return;
  uint8_t* page = lookup_page(cv, b, pg, h == 0 && threadIdx.x == 0);
  if (!page) return;
  uint4* kdst = (uint4*)(page + (size_t)h * BF16_HEAD_BYTES);
  uint4* vdst = kdst + PAGE * D * 2 / 16;
  const int nt = (hist - t0) < PAGE ? hist - t0 : PAGE;
  const size_t head = (size_t)(b * cv.Hkv + h);
  const uint4* ks = (const uint4*)(K + (head * (size_t)n + SINK + t0) * D);
  const uint4* vs = (const uint4*)(V + (head * (size_t)n + SINK + t0) * D);
  for (int i = threadIdx.x; i < nt * 16; i += blockDim.x) {
    kdst[i] = ks[i];
    vdst[i] = vs[i];
  }
}

// One token per request appended to a BF16-history cache (the baseline's
// layout: history pages of unrotated bf16 K and V rows, no quantisation).  As
// in the INT2 append, a full recent window first moves its oldest token (ring
// slot hist % 256) into history slot hist; then the new token takes sink slot
// L (L < 64) or ring slot (L - 64) % 256.  One CTA of 256 threads per request,
// 16-byte copies; a missing history page leaves the request unchanged.
__global__ void __launch_bounds__(256) append_bf16_kernel(CacheView cv, const __nv_bfloat16* __restrict__ k,
                                                          const __nv_bfloat16* __restrict__ v) {
  const int b = blockIdx.x, Hkv = cv.Hkv;
  const int L = cv.seq_lens[b], H = cv.hist_lens[b];
  const int recent = L > SINK ? L - SINK - H : 0;
  const bool demote = recent >= RECENT;
  const int rows = Hkv * 2 * (D * 2 / 16);  // uint4 copies per token: every kv head, K and V
  if (demote) {
    uint8_t* page = lookup_page(cv, b, H / PAGE, threadIdx.x == 0);
    if (!page) return;  // uniform: every thread sees the same table entry
    const int slot = H % RECENT, row = H % PAGE;
    for (int i = threadIdx.x; i < rows; i += blockDim.x) {
      const int h = i / 32, isv = (i / 16) & 1, c = i % 16;
      const size_t src = ((size_t)(b * Hkv + h) * RECENT + slot) * D;
      const uint4* from = (const uint4*)((isv ? cv.ring_v : cv.ring_k) + src) + c;
      uint4* to = (uint4*)(page + (size_t)h * BF16_HEAD_BYTES + (size_t)isv * PAGE * D * 2 + (size_t)row * D * 2) + c;
      *to = *from;
    }
  }
  __syncthreads();  // the demoted slot is the one the new token takes when the window is full
  const bool in_sink = L < SINK;
  for (int i = threadIdx.x; i < rows; i += blockDim.x) {
    const int h = i / 32, isv = (i / 16) & 1, c = i % 16;
    const size_t head = (size_t)b * Hkv + h;
    const size_t dst = in_sink ? (head * SINK + L) * D : (head * RECENT + (L - SINK) % RECENT) * D;
    uint4* to = (uint4*)((isv ? (in_sink ? cv.sink_v : cv.ring_v) : (in_sink ? cv.sink_k : cv.ring_k)) + dst) + c;
    *to = *((const uint4*)((isv ? v : k) + head * D) + c);
  }
  if (threadIdx.x == 0) {
    cv.seq_lens[b] = L + 1;
    if (demote) cv.hist_lens[b] = H + 1;
  }
}

__global__ void import_set_lengths_kernel(int32_t* seq, int32_t* hist, int B, int n) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= B) return;
  if (seq[b] != 0) return;
  seq[b] = n;
  hist[b] = n > SINK + RECENT ? n - SINK - RECENT : 0;
}

// --------------------------------------------------------------- test hooks
// grid = ceil(n / 64), block 128: each CTA quantises up to 64 rotated vectors.
__global__ void __launch_bounds__(128) quantize_hook_kernel(const float* __restrict__ x, int n,
                                                            int g, float clip, QThr th, int which,
                                                            uint8_t* __restrict__ codes,
                                                            __half2* __restrict__ sz) {
  __shared__ float red[8];
  __shared__ __align__(16) uint32_t kwords[PAGE * 8];
  __shared__ __align__(16) uint32_t vwords[D * 4];
  const int j = threadIdx.x;
  const int i0 = blockIdx.x * PAGE;
  const int cnt = (n - i0) < PAGE ? n - i0 : PAGE;
  const int NG = D / g;
  for (int i = j; i < PAGE * 8; i += 128) kwords[i] = 0u;
  for (int i = j; i < D * 4; i += 128) vwords[i] = 0u;
  __syncthreads();
  for (int t = 0; t < cnt; ++t) {
    const float y = x[(size_t)(i0 + t) * D + j];
    quant_pack(y, j, g, clip, th, red, 1, which == 1, t, kwords + t * 8, vwords,
               sz + (size_t)(i0 + t) * NG);
  }
  __syncthreads();
  if (which == 0) {
    for (int i = j; i < cnt * 8; i += 128) ((uint32_t*)codes)[(size_t)i0 * 8 + i] = kwords[i];
  } else {
    for (int i = j; i < D * 4; i += 128) ((uint32_t*)codes)[(size_t)blockIdx.x * 512 + i] = vwords[i];
  }
}

// grid = n, block 128: y = x·R, thread j = output channel j
__global__ void __launch_bounds__(128) debug_rotate_kernel(const float* __restrict__ R,
                                                           const __nv_bfloat16* __restrict__ x,
                                                           float* __restrict__ y) {
  __shared__ float xs[D];
  const int j = threadIdx.x;
  xs[j] = __bfloat162float(x[(size_t)blockIdx.x * D + j]);
  __syncthreads();
  float acc = 0.f;
#pragma unroll 8
  for (int i = 0; i < D; ++i) acc = fmaf(xs[i], __ldg(R + i * D + j), acc);
  y[(size_t)blockIdx.x * D + j] = acc;
}

}  // namespace

cudaError_t launch_append(const CacheView& cv, const LayerRot& rot, const __nv_bfloat16* k,
                          const __nv_bfloat16* v, int B, int do_append, int* req_counter,
                          cudaStream_t st, Profiler* prof) {
  prof_begin(prof, OSCAR_KERNEL_APPEND, st);
  const cudaError_t e =
      launch_pdl(append_kernel, dim3(B * cv.Hkv, 2), dim3(512), 0, st, cv, rot, k, v, do_append, req_counter);
  prof_end(prof, OSCAR_KERNEL_APPEND, st);
  return e;
}

cudaError_t launch_step(const CacheView& cv, const LayerRot& rot, const __nv_bfloat16* k,
                        const __nv_bfloat16* v, int B, int* req_counter, const DecodeArgs& a,
                        cudaStream_t st, Profiler* prof) {
  prof_begin(prof, OSCAR_KERNEL_STEP, st);
  const cudaError_t e =
      launch_pdl(step_kernel, dim3(B * cv.Hkv, 3), dim3(512), 0, st, cv, rot, k, v, req_counter, a);
  prof_end(prof, OSCAR_KERNEL_STEP, st);
  return e;
}

cudaError_t launch_append_bf16(const CacheView& cv, const __nv_bfloat16* k, const __nv_bfloat16* v, int B,
                               cudaStream_t st, Profiler* prof) {
  prof_begin(prof, OSCAR_KERNEL_APPEND, st);
  append_bf16_kernel<<<B, 256, 0, st>>>(cv, k, v);
  prof_end(prof, OSCAR_KERNEL_APPEND, st);
  return cudaGetLastError();
}

cudaError_t launch_import(const CacheView& cv, const LayerRot& rot, const __nv_bfloat16* K,
                          const __nv_bfloat16* V, int B, int n, int bf16_history,
                          cudaStream_t st, Profiler* prof) {
  prof_begin(prof, OSCAR_KERNEL_IMPORT, st);
  import_window_kernel<<<B * cv.Hkv, 256, 0, st>>>(cv, K, V, n);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int hist = n > SINK + RECENT ? n - SINK - RECENT : 0;
  const int pages = (hist + PAGE - 1) / PAGE;
  if (pages > 0) {
    dim3 grid(B * cv.Hkv, pages);
    if (bf16_history)
      import_bf16_pages_kernel<<<grid, 256, 0, st>>>(cv, K, V, n);
    else
      import_int2_pages_kernel<<<grid, 256, 0, st>>>(cv, rot, K, V, n);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  import_set_lengths_kernel<<<(B + 127) / 128, 128, 0, st>>>(cv.seq_lens, cv.hist_lens, B, n);
  prof_end(prof, OSCAR_KERNEL_IMPORT, st);
  return cudaGetLastError();
}

cudaError_t launch_quantize_hook(const float* x, int n, int g, float clip, int which, float thr_lo,
                                 float thr_hi, uint8_t* codes, __half2* sz, cudaStream_t st) {
  QThr th;
  th.lo = thr_lo;
  th.hi = thr_hi;
  quantize_hook_kernel<<<(n + PAGE - 1) / PAGE, 128, 0, st>>>(x, n, g, clip, th, which, codes, sz);
  return cudaGetLastError();
}

cudaError_t launch_debug_rotate(const float* R, const __nv_bfloat16* x, float* y, int n,
                                cudaStream_t st) {
  debug_rotate_kernel<<<n, 128, 0, st>>>(R, x, y);
  return cudaGetLastError();
}

}  // namespace oscar
