// INT2 history decode with a CTA-wide ring of page stages (sm_103a): the
// default decode kernel.
//
// The computation is the decode paragraph under the pipeline figure
// "从离线校准到在线推理的pipeline" of "超越TurboQuant：Together AI把2-bit KV Cache推向
// 真实服务": the INT2 history is unpacked, dequantised with its scale / zero
// point and accumulated in floating point (mma.sync tensor cores, page math in
// oscar_pagemath.cuh), the BF16 sink/recent segment is attended separately,
// and the parts are merged by online softmax (merge_kernel).
//
// Work: the history items of make_sched (one (request, kv head, S pages)
// item per resident CTA while items stay small; more, balanced through the
// work counter, beyond that), then the BF16 window chunks (64 tokens each) as
// single-warp jobs taken from a second counter by whichever warps finish
// their history first.
//
// Within an item the CTA's four warps share one ring of 16 page stages:
//   * page i of the item goes to stage i % 16; all of the first 16 are
//     copied as the item starts (before the wait on the query rotation);
//   * a warp takes the next unit (a pair of pages at G <= 4, else one page)
//     from a shared counter, so the four warps finish within one unit of
//     each other however the pages arrive;
//   * after its unit a warp copies pages i + 16 into the stages it freed.
// At most four units are in flight and a ring turn is eight pairs (or 16
// pages), so page i + 16 is always copied before any warp waits for it: a
// wait on the stage's phase parity is unambiguous.
#include "oscar_internal.cuh"
#include "oscar_pagemath.cuh"
#include "oscar_window.cuh"

namespace oscar {
namespace {

constexpr int RW = DEC_NW;   // warps per CTA
constexpr int RS = 16;       // ring stages
constexpr int RPIDS = 256;   // page ids of an item kept in shared memory (later ones read from global)

struct RingLayout {
  int stage_bytes, off_stage, off_mbar, off_qpk, off_pid, off_ctl, off_pre, off_red, total;
};

__host__ __device__ inline RingLayout ring_layout(int head_bytes, int B, int G) {
  RingLayout L;
  L.stage_bytes = (head_bytes + 127) & ~127;
  int o = 0;
  L.off_stage = o;
  int st = RS * L.stage_bytes;
  const int wo_bytes = RW * MAX_G * D * 4 + 2 * RW * MAX_G * 4;  // the warp results alias the stages
  if (st < wo_bytes) st = wo_bytes;
  o += (st + 127) & ~127;
  L.off_mbar = o;
  o += RS * 8;
  L.off_qpk = o;
  o += G * QPACK_BYTES;
  L.off_pid = (o + 15) & ~15;
  o = L.off_pid + RPIDS * 4;
  L.off_ctl = o;  // [0] next item, [1] abort, [2] next unit, [4..4+RS) stage uses, [4+RS..4+2RS) issued this item
  o += (4 + 2 * RS) * 4;
  L.off_pre = (o + 15) & ~15;
  o = L.off_pre + (((B + 1) * 4 + 15) & ~15);
  L.off_red = o;
  o += 2 * RW * 4;
  L.total = o;
  return L;
}

// One BF16 window chunk (64 tokens) of (b, kvh) by one warp, written as the
// chunk's partial record.
__device__ __forceinline__ void ring_window_chunk(const DecodeArgs& a, int b, int kvh, int ch, int slot, int lane) {
  const CacheView& cv = a.cv;
  const int gid = lane >> 2, tq = lane & 3, G = cv.G, Hkv = cv.Hkv;
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
  if (ch == 0) {
    valid = nsink >= 64 ? ~0ull : ((1ull << nsink) - 1ull);
    Kb = cv.sink_k + head * SINK * D;
    Vb = cv.sink_v + head * SINK * D;
  } else {
    const int s0 = 64 * (ch - 1);
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int t = lane + 32 * half;
      const bool v = ((s0 + t - h0 + RECENT) % RECENT) < recent;
      valid |= (uint64_t)__ballot_sync(0xffffffffu, v) << (32 * half);
    }
    Kb = cv.ring_k + (head * RECENT + s0) * D;
    Vb = cv.ring_v + (head * RECENT + s0) * D;
  }
  if (valid) bf16_span_mma<false>(S, Kb, Vb, valid, lane, 0, 4);
#pragma unroll
  for (int hc = 0; hc < 2; ++hc) {
    S.l[hc] += __shfl_xor_sync(0xffffffffu, S.l[hc], 4);
    S.l[hc] += __shfl_xor_sync(0xffffffffu, S.l[hc], 8);
    S.l[hc] += __shfl_xor_sync(0xffffffffu, S.l[hc], 16);
  }
#pragma unroll
  for (int hc = 0; hc < 2; ++hc) {
    const int n = 2 * tq + hc;
    if (n < G) {
      float* rec = a.part + ((size_t)slot * G + n) * PART_STRIDE;
      if (gid == 0) {
        rec[0] = S.m[hc];
        rec[1] = S.l[hc];
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        rec[PART_O + 16 * gid + 2 * j] = S.oacc[j][hc];
        rec[PART_O + 16 * gid + 2 * j + 1] = S.oacc[j][hc + 2];
      }
    }
  }
}

// PAIR: units of two pages as two softmax streams per tile (G <= 4);
// otherwise one page per unit (any G).
template <int NG, bool PAIR>
__global__ void __launch_bounds__(RW * 32, NG == 1 ? 3 : 2) decode_ring_kernel(DecodeArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  const CacheView& cv = a.cv;
  const int G = cv.G, Hkv = cv.Hkv;
  const RingLayout L = ring_layout(cv.head_bytes, a.B, G);
  uint64_t* mbar = (uint64_t*)(smem + L.off_mbar);
  uint8_t* qpk = smem + L.off_qpk;
  int* pid_s = (int*)(smem + L.off_pid);
  int* ctl = (int*)(smem + L.off_ctl);
  int* uses = ctl + 4;        // completed uses of each stage before the current item
  int* issued = ctl + 4 + RS;  // pages copied into each stage during the current item
  int* pre = (int*)(smem + L.off_pre);
  int* red = (int*)(smem + L.off_red);
  float* wm = (float*)(smem + L.off_stage);
  float* wl = wm + RW * MAX_G;
  float* wo = wl + RW * MAX_G;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, gid = lane >> 2, tq = lane & 3;
  const uint32_t hb = (uint32_t)cv.head_bytes;

  pdl_launch_dependents();  // merge_kernel may be scheduled as CTAs of this grid retire
  if (tid < RS) {
    mbar_init(&mbar[tid], 1);
    uses[tid] = 0;
  }
  if (tid == 0) ctl[1] = 0;
  fence_proxy_async();
  __syncthreads();
  // history lengths and page tables come from earlier stream work: readable
  // before the wait on the query rotation
  const Sched sc = make_sched(cv.hist_lens, a.B, Hkv, a.target_items, a.resident, cv.head_bytes, pre, red, true);
  bool waited = false;
  int it = blockIdx.x;  // first item static, later ones from the work counter

  while (it < sc.n_hist) {
    int b, kvh, jj;
    hist_item_coords(it, pre, a.B, Hkv, cv.hist_lens, sc.S, b, kvh, jj);
    const int hist_b = cv.hist_lens[b];
    const int pages_b = (hist_b + PAGE - 1) / PAGE;
    const int p0 = jj * sc.S;
    const int p1 = p0 + sc.S < pages_b ? p0 + sc.S : pages_b;
    const int n = p1 - p0;
    const int32_t* ptab = cv.page_table + (size_t)b * cv.max_pages_per_req + p0;
    for (int i = tid; i < n && i < RPIDS; i += RW * 32) pid_s[i] = __ldg(ptab + i);
    if (tid == 0) ctl[2] = 0;
    if (tid < RS) issued[tid] = 0;
    __syncthreads();
    auto pid_at = [&](int i) { return i < RPIDS ? pid_s[i] : __ldg(ptab + i); };
    auto issue = [&](int i) {  // one lane: page i of the item into stage i % RS
      const int s = i & (RS - 1);
      const int pid = pid_at(i);
      atomicAdd(&issued[s], 1);
      if (pid >= 0 && pid < cv.num_pages) {
        mbar_expect_tx(&mbar[s], hb);
        bulk_g2s(smem + L.off_stage + (size_t)s * L.stage_bytes,
                 cv.pool + (size_t)pid * cv.page_bytes + (size_t)kvh * hb, hb, &mbar[s]);
      } else {
        record_error(cv.err, pid < 0 ? OSCAR_ERR_NO_PAGE : OSCAR_ERR_RANGE);
        mbar_expect_tx(&mbar[s], 0u);
      }
    };
    // the first ring turn, spread over the warps' lane 0
    if (lane == 0)
      for (int i = warp; i < n && i < RS; i += RW) issue(i);
    if (!waited) {
      pdl_wait();  // the packed query (prep / step kernel) is ready from here on
      waited = true;
    }
    // the kv head's G packed query records, coalesced 16-byte loads by warp 0
    if (warp == 0) {
      const uint4* src = (const uint4*)(a.qpack + ((size_t)b * cv.Hq + kvh * G) * QPACK_BYTES);
      for (int e = lane; e < G * QPACK_BYTES / 16; e += 32) ((uint4*)qpk)[e] = __ldcg(src + e);
    }
    __syncthreads();
    Int2State<NG> S;
#pragma unroll
    for (int j = 0; j < 8; ++j) S.oacc[j][0] = S.oacc[j][1] = S.oacc[j][2] = S.oacc[j][3] = 0.f;
    {
      // B column gid carries head gid (PAIR: head gid & 3 in both halves)
      const int qh = PAIR ? (gid & 3) : gid;
      const bool qv = qh < G;
      const __half* qbh = (const __half*)(qpk + (qv ? qh : 0) * QPACK_BYTES);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        S.bq[kk][0] = qv ? *(const unsigned int*)(qbh + 16 * kk + 2 * tq) : 0u;
        S.bq[kk][1] = qv ? *(const unsigned int*)(qbh + 16 * kk + 8 + 2 * tq) : 0u;
      }
#pragma unroll
      for (int hc = 0; hc < 2; ++hc) {
        const int hn = PAIR ? ((2 * tq + hc) & 3) : 2 * tq + hc;
        const bool hv = hn < G;
        const uint8_t* r = qpk + (hv ? hn : 0) * QPACK_BYTES;
        S.m[hc] = PAIR ? -1e30f : -INFINITY;
        S.l[hc] = 0.f;
        // subnormal codes: 2^24 times the record's logit scale, no logit offset
        S.ka[hc] = hv ? *(const float*)(r + QPACK_ALPHA) * 16777216.f : 0.f;
#pragma unroll
        for (int gr = 0; gr < NG; ++gr) {
          float ps = 0.f;
#pragma unroll
          for (int k = gr * (4 / NG); k < (gr + 1) * (4 / NG); ++k) ps += hv ? ((const float*)(r + QPACK_PSUM))[k] : 0.f;
          S.bs[hc][gr] = 0.f;
          S.zs[hc][gr] = 0.f;
          S.kb[hc][gr] = 0.f;
          S.kg[hc][gr] = ps * LOG2E * INV_SQRT_D;
        }
      }
    }
    const uint32_t mA = gid < 4 ? 0xffffffffu : 0u;  // PAIR: B columns 0..3 belong to page A
    const int units = PAIR ? (n + 1) / 2 : n;
    auto nvalid = [&](int i) {  // valid tokens of page i of the item (0 for a bad page id)
      const int pid = pid_at(i);
      if (pid < 0 || pid >= cv.num_pages) return 0;
      const int p = p0 + i;
      return (p == pages_b - 1) ? hist_b - p * PAGE : PAGE;
    };
    while (true) {
      int u = 0;
      if (lane == 0) u = ctl[1] ? units : atomicAdd(&ctl[2], 1);
      u = __shfl_sync(0xffffffffu, u, 0);
      if (u >= units) break;
      const int ia = PAIR ? 2 * u : u;
      const bool hasB = PAIR && ia + 1 < n;
      const int sa = ia & (RS - 1), sb = (ia + 1) & (RS - 1);
      const uint32_t pha = (uint32_t)(uses[sa] + (ia >> 4)) & 1u;
      bool ok;
      if (hasB)
        ok = mbar_wait2(&mbar[sa], pha, &mbar[sb], (uint32_t)(uses[sb] + ((ia + 1) >> 4)) & 1u);
      else
        ok = mbar_wait(&mbar[sa], pha);
      if (!__all_sync(0xffffffffu, ok)) {
        if (lane == 0) {
          record_error(cv.err, OSCAR_ERR_TIMEOUT);
          atomicExch(&ctl[1], 1);
        }
        break;
      }
      const uint8_t* sta = smem + L.off_stage + (size_t)sa * L.stage_bytes;
      if constexpr (PAIR) {
        const uint8_t* stb = hasB ? smem + L.off_stage + (size_t)sb * L.stage_bytes : sta;
        const int nva = nvalid(ia), nvb = hasB ? nvalid(ia + 1) : 0;
        // one (masked) variant for full and partial pages keeps the
        // unrolled loop body small enough for the instruction cache
        int2_pair_mma<NG, false>(S, sta, nva, stb, nvb, hasB, lane, mA);
      } else {
        const int nv = nvalid(ia);
        if (nv == PAGE)
          int2_page_mma<NG, true, true>(S, sta, nv, lane);
        else if (nv > 0)
          int2_page_mma<NG, false, true>(S, sta, nv, lane);
      }
      __syncwarp();
      // the stages' generic-proxy reads have completed (their values were
      // consumed before __syncwarp): no proxy fence is needed
      if (lane == 0) {
        if (ia + RS < n) issue(ia + RS);
        if (hasB && ia + 1 + RS < n) issue(ia + 1 + RS);
      }
    }
#pragma unroll
    for (int hc = 0; hc < 2; ++hc) {
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        S.l[hc] += __shfl_xor_sync(0xffffffffu, S.l[hc], o);
#pragma unroll
        for (int gr = 0; gr < NG; ++gr) S.zs[hc][gr] += __shfl_xor_sync(0xffffffffu, S.zs[hc][gr], o);
      }
    }
    if constexpr (PAIR) merge_pair_streams<NG>(S);
    __syncthreads();  // every warp is past the ring
    const bool aborted = ctl[1] != 0;
    if (aborted && tid < RS && issued[tid] > 0) {
      // copies still in flight land before the stages are reused or the CTA
      // exits: the stage's last use, after the one before it
      const int ul = uses[tid] + issued[tid] - 1;
      if (ul > 0) mbar_wait(&mbar[tid], (uint32_t)(ul - 1) & 1u);
      mbar_wait(&mbar[tid], (uint32_t)ul & 1u);
    }
    __syncthreads();  // results may alias the stages
#pragma unroll
    for (int hc = 0; hc < 2; ++hc) {
      const int hn = 2 * tq + hc;
      if (hn < G) {
        if (gid == 0) {
          wm[warp * MAX_G + hn] = S.m[hc];
          wl[warp * MAX_G + hn] = S.l[hc];
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int gr = j / (8 / NG);
          const float z = S.zs[hc][gr];
          // o' = 2^16 * O + sum p z  (P·s carried 2^(8 - E), the codes 2^(E - 24))
          wo[(warp * MAX_G + hn) * D + 16 * j + gid] = fmaf(S.oacc[j][hc], 65536.f, z);
          wo[(warp * MAX_G + hn) * D + 16 * j + 8 + gid] = fmaf(S.oacc[j][hc + 2], 65536.f, z);
        }
      }
    }
    __syncthreads();
    cta_combine_write(a, wm, wl, wo, it);
    if (tid < RS) uses[tid] += issued[tid];
    if (aborted) break;
    __syncthreads();
    if (tid == 0) ctl[0] = (int)gridDim.x + atomicAdd(a.counter, 1);
    __syncthreads();
    it = ctl[0];
  }
  // ---- BF16 window chunks: single-warp jobs for the warps done first
  if (!waited) {
    pdl_wait();  // the window contents and q come from earlier stream work
    waited = true;
  }
  if (!ctl[1]) {
    while (true) {
      int c = 0;
      if (lane == 0) c = atomicAdd(a.counter + 1, 1);
      c = __shfl_sync(0xffffffffu, c, 0);
      if (c >= sc.n_win) break;
      const int bk = c / WIN_CHUNKS, ch = c % WIN_CHUNKS;
      ring_window_chunk(a, bk / Hkv, bk % Hkv, ch, sc.n_hist + c, lane);
    }
  }
}

template <int NG, bool PAIR>
cudaError_t launch_ring_t(const DecodeArgs& a, int grid, cudaStream_t st) {
  const RingLayout L = ring_layout(a.cv.head_bytes, a.B, a.cv.G);
  if ((L.off_mbar % 8) || (L.off_stage % 128) || (L.off_qpk % 16) || (L.off_pid % 16)) return cudaErrorInvalidValue;
  static int limit[MAX_DEVICES];
  const cudaError_t e = raise_smem_limit(decode_ring_kernel<NG, PAIR>, limit, L.total);
  if (e != cudaSuccess) return e;
  return launch_pdl(decode_ring_kernel<NG, PAIR>, dim3(grid), dim3(RW * 32), L.total, st, a);
}

template <int NG, bool PAIR>
int ring_occupancy_t(const DecodeArgs& a) {
  static int cached_smem[MAX_DEVICES], cached_occ[MAX_DEVICES];
  const RingLayout L = ring_layout(a.cv.head_bytes, a.B, a.cv.G);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) {
    (void)cudaGetLastError();
    return 0;
  }
  if (cached_smem[dev] == L.total) return cached_occ[dev];
  static int limit[MAX_DEVICES];
  int n = 0;
  if (raise_smem_limit(decode_ring_kernel<NG, PAIR>, limit, L.total) != cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_ring_kernel<NG, PAIR>, RW * 32, L.total) !=
          cudaSuccess) {
    (void)cudaGetLastError();
    return 0;
  }
  cached_occ[dev] = n;
  cached_smem[dev] = L.total;
  return n;
}

}  // namespace

cudaError_t launch_decode_ring(const DecodeArgs& a, int grid, cudaStream_t st) {
  const bool pair = a.impl == 3;
  if (pair) {
    if (a.cv.NG == 1) return launch_ring_t<1, true>(a, grid, st);
    if (a.cv.NG == 2) return launch_ring_t<2, true>(a, grid, st);
    return launch_ring_t<4, true>(a, grid, st);
  }
  if (a.cv.NG == 1) return launch_ring_t<1, false>(a, grid, st);
  if (a.cv.NG == 2) return launch_ring_t<2, false>(a, grid, st);
  return launch_ring_t<4, false>(a, grid, st);
}

int decode_ring_ctas_per_sm(const DecodeArgs& a) {
  const bool pair = a.impl == 3;
  if (pair) return a.cv.NG == 1 ? ring_occupancy_t<1, true>(a) : a.cv.NG == 2 ? ring_occupancy_t<2, true>(a)
                                                                                : ring_occupancy_t<4, true>(a);
  return a.cv.NG == 1 ? ring_occupancy_t<1, false>(a) : a.cv.NG == 2 ? ring_occupancy_t<2, false>(a)
                                                                      : ring_occupancy_t<4, false>(a);
}

}  // namespace oscar
