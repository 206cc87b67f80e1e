// Internal device helpers and kernel entry points of liboscar (sm_103a).
//
// Sources, cited by page title and section:
//  [News] "Together AI 开源 OSCAR：一种面向长上下文 LLM 服务的注意力感知 2 位 KV 缓存量化系统"
//  [Blog] "超越TurboQuant：Together AI把2-bit KV Cache推向真实服务"
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "../../include/oscar.h"

namespace oscar {

constexpr int D = 128;       // head_dim
constexpr int PAGE = 64;     // tokens per page
constexpr int SINK = 64;     // BF16 sink tokens   [News, "服务系统：混合精度缓存布局"]
constexpr int RECENT = 256;  // BF16 recent tokens [News, "服务系统：混合精度缓存布局"]
constexpr int MAX_G = 8;     // query heads per KV head handled by one mma column tile
constexpr int PART_STRIDE = D + 4;  // partial record per head: m, l, 2 pad, o[128] (o 16-byte aligned)
constexpr int PART_O = 4;            // offset of o in a partial record
constexpr int MAX_TARGET_ITEMS = 2048;
constexpr int QPACK_BYTES = 320;  // packed query record per (request, query head)
constexpr int QPACK_CB_BYTES = 576;  // the same with a Lloyd-Max codebook (two B operands)
// Per-head codebook record (floats): the levels of the normalised value t are
// {1.5-b, 1.5-a, 1.5+a, 1.5+b}; a code is [t > lo] + [t >= 1.5] + [t > hi]
// with lo/hi = 1.5 -/+ (a+b)/2; c0, alpha = b - a and beta_half = (a + b)/2
// give level(code) = c0 + alpha*bit0 + 2*beta_half*bit1.  Uniform: a = 0.5, b = 1.5.
constexpr int CB_WORDS = 8;
enum { CB_A = 0, CB_B, CB_LO, CB_HI, CB_C0, CB_ALPHA, CB_BETA_HALF };
constexpr int WIN_BYTES_PER_HEAD = (SINK + RECENT) * D * 2 * 2;  // K and V
constexpr int BF16_HEAD_BYTES = PAGE * D * 2 * 2;
constexpr float LOG2E = 1.4426950408889634f;
constexpr float LN2 = 0.6931471805599453f;
constexpr float INV_SQRT_D = 0.08838834764831845f;  // 1/sqrt(128)

__host__ __device__ constexpr int int2_head_bytes(int g) { return 4096 + PAGE * (D / g) * 8; }
__host__ __device__ constexpr int off_k_sz() { return 4096; }
__host__ __device__ constexpr int off_v_sz(int g) { return 4096 + PAGE * (D / g) * 4; }

// Per-layer rotation tables on the device (owned by the context).
// R_V in mma.m16n8k16 A-fragment order, for o = o'·R_V^T on tensor cores
// (A = R_V, rows = output channels, columns = input channels): per kv head,
// part (0: fp16 of R_V, 1: fp16 of the remainder R_V - part 0), m-tile mt,
// k-step ks and lane (gid, tq), the four words a0..a3 hold
// R_V[16mt+gid(+8)][16ks+2tq(+8) +0/+1], lower column in the low half.
constexpr int RV_FRAG_WORDS = 2 * 8 * 8 * 32 * 4;  // per kv head: 64 KB

__host__ __device__ __forceinline__ int rv_frag_index(int part, int mt, int ks, int lane) {
  return (((part * 8 + mt) * 8 + ks) * 32 + lane) * 4;
}

// Per-layer rotation table, composed in fp64 on the host from the eigenbases:
// R_K = rotation(U_K, mode) and R_V = rotation(U_V, mode) in fp32 for the
// demotion and the query, R_V again as fp16 high/low fragments for the
// decode's output and as fp32 R_V^T for the prefill's output.
struct LayerRot {
  const float* R_K;         // [Hkv][128][128]  k' = k·R_K, q' = q·R_K
  const float* R_V;         // [Hkv][128][128]  v' = v·R_V
  const uint32_t* RV_frag;  // [Hkv][RV_FRAG_WORDS]  o = o'·R_V^T
  const float* RVt;         // [Hkv][128][128]  R_V^T, row i = column i of R_V (coalesced un-rotation)
  const float* clip_k;      // [Hkv]
  const float* clip_v;      // [Hkv]
  const float* cb;          // [2][Hkv][CB_WORDS] codebook records, K then V
  int mode;
};

// Everything a kernel needs to know about the cache and the configuration.
struct CacheView {
  uint8_t* pool;
  const int32_t* page_table;
  __nv_bfloat16* sink_k;
  __nv_bfloat16* sink_v;
  __nv_bfloat16* ring_k;
  __nv_bfloat16* ring_v;
  int32_t* seq_lens;
  int32_t* hist_lens;
  int Hq, Hkv, G, g, NG;
  int max_pages_per_req, num_pages;
  long long page_bytes;  // bytes per page (all heads)
  int head_bytes;        // bytes of one head's block
  int* err;
};

// Release/acquire fence at GPU scope (lighter than a sequentially consistent one).
__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;\n" ::: "memory"); }

// atomicAdd with acquire-release semantics at GPU scope.
__device__ __forceinline__ int atomic_add_acq_rel_gpu(int* p, int v) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;\n" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

// 2^n for -126 <= n <= 127, from the exponent bits (the cold prologues stay
// short: no library call).
__device__ __forceinline__ float pow2i(int n) { return __uint_as_float((uint32_t)(127 + n) << 23); }

__device__ __forceinline__ void record_error(int* err, int code) {
  if (err) atomicCAS(err, 0, code);
}

// ---------------------------------------------------------------- layouts
// K codes, token-major: channel c = 64A+16B+8C+2D+E -> word 2D+A, bit 16E+2(2B+C).
__host__ __device__ __forceinline__ int k_word(int c) { return 2 * ((c >> 1) & 3) + (c >> 6); }
__host__ __device__ __forceinline__ int k_bit(int c) {
  return 16 * (c & 1) + 2 * (2 * ((c >> 4) & 3) + ((c >> 3) & 1));
}
// V codes, channel-major: token slot t = 16S+8A+2T+E -> word T, bit 16E+2(2S+A).
__host__ __device__ __forceinline__ int v_word(int t) { return (t >> 1) & 3; }
__host__ __device__ __forceinline__ int v_bit(int t) {
  return 16 * (t & 1) + 2 * (2 * (t >> 4) + ((t >> 3) & 1));
}

// ------------------------------------------------------- 128-thread groups
// A "group" is 128 consecutive threads (4 full warps) holding one 128-channel
// vector, one channel per thread.  Named barrier `bar` (1..15) syncs it.
__device__ __forceinline__ void group_sync(int bar) {
  asm volatile("bar.sync %0, 128;" ::"r"(bar) : "memory");
}

__device__ __forceinline__ int bitrev7(int j) { return (int)(__brev((unsigned)j) >> 25); }

// --------------------------------------------------------------- quantiser
// [Blog, pipeline figure paragraph: rotate -> clip -> quantize -> pack].
// Each step is one IEEE float32 operation rounded to nearest even; the scale
// and zero point are fp16 (round to nearest even, saturated at +-65504).
__device__ __forceinline__ __half half_rn_sat(float x) {
  __half h = __float2half_rn(x);
  if (__hisinf(h)) h = __float2half_rn(x > 0.f ? 65504.f : -65504.f);
  return h;
}

struct QParams {
  __half s, z;
};

__device__ __forceinline__ QParams quant_params(float mn, float mx, float clip) {
  const float mx_c = __fmul_rn(clip, mx);
  const float mn_c = __fmul_rn(clip, mn);
  const float s32 = __fdiv_rn(__fsub_rn(mx_c, mn_c), 3.0f);
  QParams p;
  p.s = half_rn_sat(s32);
  p.z = half_rn_sat(mn_c);
  return p;
}

// Thresholds of the codes on t = (x - z)/s: the nearest of the four levels,
// ties to the even code.  For the uniform levels {0, 1, 2, 3} (lo = 0.5,
// hi = 2.5) this is clamp(rint(t), 0, 3) for every float t.
struct QThr {
  float lo, hi;
};

__device__ __forceinline__ QThr quant_thr(const float* cb_rec) {
  QThr q;
  q.lo = __ldg(cb_rec + CB_LO);
  q.hi = __ldg(cb_rec + CB_HI);
  return q;
}

__device__ __forceinline__ uint32_t quant_code(float x, QParams p, QThr th) {
  const float sf = __half2float(p.s);
  if (sf == 0.f) return 0u;
  const float t = __fdiv_rn(__fsub_rn(x, __half2float(p.z)), sf);
  return (uint32_t)(t > th.lo) + (uint32_t)(t >= 1.5f) + (uint32_t)(t > th.hi);
}

// min and max over each group of g consecutive channels (g = 32, 64, 128),
// one channel per thread of a 128-thread group.  red: 8 floats of smem.
__device__ __forceinline__ void group_minmax(float x, int j, int g, float* red, int bar,
                                             float& mn, float& mx) {
  float a = x, b = x;
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
    b = fminf(b, __shfl_xor_sync(0xffffffffu, b, o));
  }
  if (g == 32) {
    mx = a;
    mn = b;
    return;
  }
  const int w = j >> 5;
  if ((j & 31) == 0) {
    red[w] = a;
    red[4 + w] = b;
  }
  group_sync(bar);
  const int wpg = g >> 5;
  const int w0 = (w / wpg) * wpg;
  mx = red[w0];
  mn = red[4 + w0];
  for (int k = 1; k < wpg; ++k) {
    mx = fmaxf(mx, red[w0 + k]);
    mn = fminf(mn, red[4 + w0 + k]);
  }
  group_sync(bar);
}

// ------------------------------------------------------- tensor-core helpers
__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                        uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;\n" : "=r"(y) : "r"(x));
  return y;
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;\n" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}

// Two 2-bit codes -> f16x2 without a conversion instruction: the code pair at
// bit pair I of each 16-bit half of w is moved into mantissa bits 4..9 and
// OR-ed with the exponent of 1024, giving 1024 + code * 2^E(I) exactly, with
// E = {4,6,4,6,8,4,6,8}[I].  Callers fold 2^-E and the 1024 offset into the
// other operand.
// (a & m) | c in one LOP3 (both constants in registers, so the compiler does
// not split it into an AND and an OR).
__device__ __forceinline__ uint32_t and_or(uint32_t a, uint32_t m, uint32_t c) {
  uint32_t r;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;\n" : "=r"(r) : "r"(a), "r"(m), "r"(c));
  return r;
}

template <int I>
__device__ __forceinline__ uint32_t code_pair(uint32_t w) {
  constexpr uint32_t M = (I == 0 || I == 2 || I == 5) ? 0x00300030u
                         : (I == 1 || I == 3 || I == 6) ? 0x00C000C0u
                                                        : 0x03000300u;
  // w << 4 as a multiply (FMA pipe), w >> 6 as a shift
  const uint32_t src = (I <= 1) ? (w * 16u) : (I <= 4) ? w : (w >> 6);
  return and_or(src, M, 0x64006400u);
}
// One bit of each of the two codes code_pair<I> takes: bit plane P (0 = low
// bit, 1 = high bit) as 1024 + bit * 2^(E + P) in each fp16 half.
template <int I, int P>
__device__ __forceinline__ uint32_t code_plane(uint32_t w) {
  constexpr uint32_t M = ((I == 0 || I == 2 || I == 5) ? 0x00300030u
                          : (I == 1 || I == 3 || I == 6) ? 0x00C000C0u
                                                         : 0x03000300u) &
                         (P ? 0xAAAAAAAAu : 0x55555555u);
  const uint32_t src = (I <= 1) ? (w * 16u) : (I <= 4) ? w : (w >> 6);
  return and_or(src, M, 0x64006400u);
}
// Bit plane P of code pair I as an fp16 subnormal: bit * 2^(E(I) + P - 24).
template <int I, int P>
__device__ __forceinline__ uint32_t code_plane_sub(uint32_t w) {
  constexpr uint32_t M = ((I == 0 || I == 2 || I == 5) ? 0x00300030u
                          : (I == 1 || I == 3 || I == 6) ? 0x00C000C0u
                                                         : 0x03000300u) &
                         (P ? 0xAAAAAAAAu : 0x55555555u);
  const uint32_t src = (I <= 1) ? (w * 16u) : (I <= 4) ? w : (w >> 6);
  return src & M;
}
// The same code pair as an fp16 subnormal: code * 2^(E(I) - 24), one AND
// and no offset (the tensor cores take fp16 subnormals exactly).  Callers
// fold 2^(24 - E) into the other operand or the epilogue.
template <int I>
__device__ __forceinline__ uint32_t code_sub(uint32_t w) {
  constexpr uint32_t M = (I == 0 || I == 2 || I == 5) ? 0x00300030u
                         : (I == 1 || I == 3 || I == 6) ? 0x00C000C0u
                                                        : 0x03000300u;
  const uint32_t src = (I <= 1) ? (w * 16u) : (I <= 4) ? w : (w >> 6);
  return src & M;
}
// Code pair I of w, offset (1024 + code 2^E) or subnormal (code 2^(E - 24)).
template <int I, bool SUB>
__device__ __forceinline__ uint32_t code_fp16(uint32_t w) {
  if constexpr (SUB) return code_sub<I>(w);
  else return code_pair<I>(w);
}
template <int I>
__host__ __device__ constexpr int code_exp() {
  return (I == 0 || I == 2 || I == 5) ? 4 : (I == 1 || I == 3 || I == 6) ? 6 : 8;
}
__host__ __device__ __forceinline__ int code_exp_rt(int i) {
  return (i == 0 || i == 2 || i == 5) ? 4 : (i == 1 || i == 3 || i == 6) ? 6 : 8;
}

// ------------------------------------------- programmatic dependent launch
// Every hot-path kernel is launched as a programmatic dependent of the work
// before it on the stream.  A kernel waits (griddepcontrol.wait) before it
// reads anything earlier stream work may still write, and signals its own
// dependents (griddepcontrol.launch_dependents) only once their pre-wait work
// is safe: the rotation table, written synchronously by oscar_set_rotation,
// may be read before the wait.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
}

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args&&... args) {
  cudaLaunchConfig_t lc = {};
  lc.gridDim = grid;
  lc.blockDim = block;
  lc.dynamicSmemBytes = smem;
  lc.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = attr;
  lc.numAttrs = 1;
  return cudaLaunchKernelEx(&lc, kernel, std::forward<Args>(args)...);
}

// -------------------------------------------- per-device kernel attributes
// cudaFuncSetAttribute applies to the current device only, so a raised
// dynamic shared-memory limit is remembered per device ordinal: `limit` is a
// zero-initialised array of MAX_DEVICES entries owned by the caller (one per
// kernel).  The limit is only ever raised.  Concurrent callers may both set
// the attribute, which is harmless.
constexpr int MAX_DEVICES = 64;

template <typename Kernel>
cudaError_t raise_smem_limit(Kernel kernel, int* limit, int bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= MAX_DEVICES) return cudaErrorInvalidDevice;
  if (bytes <= limit[dev]) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) limit[dev] = bytes;
  return e;
}

// ----------------------------------------------------- bounded mbarrier use
__device__ __forceinline__ void mbar_init(uint64_t* bar, int count) {
  uint32_t a = (uint32_t)__cvta_generic_to_shared(bar);
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(a), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  uint32_t a = (uint32_t)__cvta_generic_to_shared(bar);
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(a), "r"(bytes)
               : "memory");
}

constexpr int WAIT_POLLS = 1 << 22;  // iteration budget of a bounded wait

// Both phases complete (the two polls are issued together); false when the
// wait ran out of its iteration budget (`polls` polls; 0 gives up at once).
__device__ __forceinline__ bool mbar_wait2(uint64_t* bar0, uint32_t phase0, uint64_t* bar1,
                                           uint32_t phase1, int polls = WAIT_POLLS) {
  const uint32_t a0 = (uint32_t)__cvta_generic_to_shared(bar0);
  const uint32_t a1 = (uint32_t)__cvta_generic_to_shared(bar1);
  uint32_t done0 = 0, done1 = 0;
  for (int it = 0; it < polls; ++it) {
    uint32_t ok0 = 1, ok1 = 1;
    if (!done0)
      asm volatile(
          "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
          " selp.u32 %0, 1, 0, p;\n}\n"
          : "=r"(ok0)
          : "r"(a0), "r"(phase0)
          : "memory");
    if (!done1)
      asm volatile(
          "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
          " selp.u32 %0, 1, 0, p;\n}\n"
          : "=r"(ok1)
          : "r"(a1), "r"(phase1)
          : "memory");
    done0 |= ok0;
    done1 |= ok1;
    if (done0 && done1) return true;
  }
  return false;
}

// Returns false when the wait ran out of its iteration budget (`polls` polls;
// 0 gives up at once).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t phase, int polls = WAIT_POLLS) {
  uint32_t a = (uint32_t)__cvta_generic_to_shared(bar);
  for (int it = 0; it < polls; ++it) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(a), "r"(phase)
        : "memory");
    if (ok) return true;
  }
  return false;
}

// Plain (non-multicast) bulk copy global -> this CTA's shared memory,
// completing on an mbarrier.  dst, src 16-byte aligned; bytes a multiple of 16.
// An L2 policy that marks lines for eviction first: a decode reads each
// history page once per call, so its copies should not displace the lines
// that stay hot (partial records, page tables, windows, query records).
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;\n" : "=l"(p));
  return p;
}
// bulk_g2s with an L2 cache policy (l2_evict_first_policy for streamed pages)
__device__ __forceinline__ void bulk_g2s_hint(void* dst, const void* src, uint32_t bytes,
                                              uint64_t* bar, uint64_t policy) {
  uint32_t d = (uint32_t)__cvta_generic_to_shared(dst);
  uint32_t b = (uint32_t)__cvta_generic_to_shared(bar);
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, "
      "[%3], %4;\n" ::"r"(d),
      "l"(src), "r"(bytes), "r"(b), "l"(policy)
      : "memory");
}
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar) {
  uint32_t d = (uint32_t)__cvta_generic_to_shared(dst);
  uint32_t b = (uint32_t)__cvta_generic_to_shared(bar);
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(
          d),
      "l"(src), "r"(bytes), "r"(b)
      : "memory");
}

__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}

// ----------------------------------------------------------- work schedule
// The decode work is a list of items: one BF16 window item per (request, kv
// head) and history items of S consecutive pages.  Every CTA of the decode
// kernel and the merge kernel derive the same list from the device-resident
// history lengths, so no host round trip is needed.
struct Sched {
  int S;            // pages per history item
  int n_hist;       // number of history items
  int n_win;        // number of window items (B * Hkv * wch)
  int wch;          // window items per (request, kv head): 5 (one per 64-token chunk) or 1
  int win_first;    // window items are handed out before history items
  long long pages;  // history pages of all (request, kv head)
};

// Automatic item sizing (resident > 0): one item per resident CTA while that
// keeps items at most auto_wave_pages() pages (per-item start and merge costs
// favour few items); beyond that, items for up to target / resident per CTA,
// at least AUTO_MIN_PAGES pages each, balanced through the work counter.  The
// automatic partition switches to the balanced one at the same size
// (use_balanced).  INT2 kernels, batch 1, one item per CTA against the
// balanced partition: 150K 34.1 / 40.7 us, 200K 41.4 / 46.4, 300K 55.7 /
// 57.8, 400K 70.0 / 68.4; the BF16-history kernel keeps 40 pages (at 200K
// one item per CTA took 136.9 us against 130.8 balanced).
constexpr int AUTO_ITEMS_PER_CTA = 4;
// Weight of one BF16 window chunk (64 tokens of one kv head) in history pages
// in decode_kernel's balanced partition.
constexpr int DEC_WIN_WEIGHT = 12;
__host__ __device__ __forceinline__ int auto_wave_pages(bool bf16_history) { return bf16_history ? 40 : 96; }
constexpr int AUTO_MIN_PAGES = 28;

// Item size granule of the one-item-per-CTA list: the page-pair kernel
// (impl 3) rounds items up to whole pairs for each of its 4 warps (8 pages):
// no item ends in a half-empty pair, and fewer items leave fewer partial
// records to merge (batch 1, 10K: step 17.2 -> 14.3 us; 100K: decode 27.3 ->
// 27.0 us, step unchanged within 0.2 us).  The one-page-per-tile kernels keep
// exact sizes (the codebook kernel measured 38.6 -> 39.3 us with 8 in one
// run, within that leg's run-to-run spread).
__host__ __device__ __forceinline__ int pages_granule(int impl) { return impl == 3 ? 8 : 1; }

// pre: smem int[B + 1]; filled with Hkv * (history items of requests < b).
// target: the most items the list may hold; resident: the decode CTAs that
// run at once, or 0 to size items for `target` items in total.  granule:
// with one item per CTA, items are a multiple of it (pages_granule()).
// wave_pages: auto_wave_pages().
// Must be called by all threads of the block.
__device__ inline Sched make_sched(const int32_t* hist_lens, int B, int Hkv, int target, int resident,
                                   int hist_item_unit_bytes, int* pre, int* red, int granule, int wave_pages) {
  const int tid = threadIdx.x;
  // total history pages (over requests), times Hkv
  int local = 0;
#pragma unroll 1
  for (int b = tid; b < B; b += blockDim.x) local += (hist_lens[b] + PAGE - 1) / PAGE;
  // block reduce (red: one int per warp)
  local = __reduce_add_sync(0xffffffffu, local);
  if ((tid & 31) == 0) red[tid >> 5] = local;
  __syncthreads();
  int total = 0;
#pragma unroll 1
  for (int w = 0; w < (int)(blockDim.x + 31) / 32; ++w) total += red[w];
  __syncthreads();
  total *= Hkv;
  Sched s;
  // items = the list size aimed for; small batches split each 320-token
  // window into its 5 chunks so that no single window item outlasts the
  // history items
  auto pages_per_item = [&](int items) {
    s.wch = (5LL * B * Hkv * 4 <= items) ? 5 : 1;
    s.n_win = B * Hkv * s.wch;
    int th = items - s.n_win;
    if (th < (items + 1) / 2) th = (items + 1) / 2;
    const int S = (total + th - 1) / th;
    return S < 1 ? 1 : S;
  };
  int S = pages_per_item(resident > 0 ? resident : target);
  if (resident > 0 && S > wave_pages) {
    S = pages_per_item(target);
    if (S < AUTO_MIN_PAGES) S = AUTO_MIN_PAGES;
  } else if (resident > 0) {
    S = (S + granule - 1) / granule * granule;
  }
  s.S = (int)S;
  if (tid == 0) {
    // per-request rounding can add up to B*Hkv items: grow S until they fit
#pragma unroll 1
    for (int iter = 0; iter < 32; ++iter) {
      long long n = 0;
#pragma unroll 1
      for (int b = 0; b < B; ++b) {
        const int pages = (hist_lens[b] + PAGE - 1) / PAGE;
        n += (long long)Hkv * ((pages + s.S - 1) / s.S);
      }
      if (n + s.n_win <= target || n <= (long long)B * Hkv) break;
      s.S += s.S / 8 > 1 ? s.S / 8 : 1;
    }
    int acc = 0;
#pragma unroll 1
    for (int b = 0; b < B; ++b) {
      pre[b] = acc;
      const int pages = (hist_lens[b] + PAGE - 1) / PAGE;
      acc += Hkv * ((pages + s.S - 1) / s.S);
    }
    pre[B] = acc;
    red[0] = s.S;
  }
  __syncthreads();
  s.S = red[0];
  __syncthreads();
  s.n_hist = pre[B];
  s.pages = total;
  s.win_first = (long long)(WIN_BYTES_PER_HEAD / s.wch) > (long long)s.S * hist_item_unit_bytes;
  return s;
}

// history item q -> (b, kvh, j); pre has B + 1 entries.
__device__ __forceinline__ void hist_item_coords(int q, const int* pre, int B, int Hkv,
                                                 const int32_t* hist_lens, int S, int& b,
                                                 int& kvh, int& j) {
  int lo = 0, hi = B - 1;
  while (lo < hi) {  // largest b with pre[b] <= q
    int mid = (lo + hi + 1) >> 1;
    if (pre[mid] <= q) lo = mid; else hi = mid - 1;
  }
  b = lo;
  const int pages = (hist_lens[b] + PAGE - 1) / PAGE;
  const int nb = (pages + S - 1) / S;
  const int r = q - pre[b];
  kvh = r / nb;
  j = r % nb;
}

// ------------------------------------------- balanced partition (tcgen05)
// The tensor-memory decode kernel runs one CTA per SM and splits the work
// evenly without a work counter.  The work is a sequence of segments, one per
// (request b, kv head) in order.  Segment (b, kvh) holds request b's history
// pages (weight 1 each), then its non-empty BF16 window chunks (chunk 0 is the
// sink, chunks 1..4 the four 64-slot quarters of the ring; weight `wch` each).
// With W the total weight and n = min(CTAs, W) CTAs taking part, CTA i takes
// the units whose position lies in [floor(i W / n), floor((i + 1) W / n)):
// never an empty range, since n <= W.  Its pages of a segment form one
// history item with partial record i + (b Hkv + kvh) (distinct over all
// (CTA, segment) pairs, because a later segment's pages never go to an
// earlier CTA); window chunk c of the segment is taken by the CTA whose range
// holds the chunk's first position and has partial record
// n + B Hkv + 5 (b Hkv + kvh) + c.  The merge derives the same list.
constexpr int WIN_CHUNKS = 5;

// Bit c set when window chunk c of a request with L tokens, hist of them in
// history, holds a valid token.
__host__ __device__ __forceinline__ unsigned window_chunk_mask(int L, int hist) {
  unsigned m = L > 0 ? 1u : 0u;
  const int recent = L > SINK ? L - SINK - hist : 0;
  if (recent > 0) {
    const int h0 = hist % RECENT;
    for (int c = 1; c < WIN_CHUNKS; ++c) {
      const int d = (64 * (c - 1) - h0 + RECENT) % RECENT;  // offset of the chunk's first slot from h0
      if (d < recent || d > RECENT - 64) m |= 1u << c;       // d > 192: the chunk wraps through h0
    }
  }
  return m;
}

struct Balanced {
  long long W;  // total weight
  int n;        // CTAs taking part (min(grid, W))
  int wch;      // weight of a window chunk
};

// pre[b] = Hkv * (weights of requests < b), pre[B] = W (smem, B + 1 entries).
// All threads of the block call it.
__device__ inline Balanced make_balanced(const int32_t* seq_lens, const int32_t* hist_lens, int B, int Hkv,
                                         int wch, int grid, long long* pre) {
  if (threadIdx.x == 0) {
    long long acc = 0;
    for (int b = 0; b < B; ++b) {
      pre[b] = acc;
      const int L = seq_lens[b], H = hist_lens[b];
      const int pages = H > 0 ? (H + PAGE - 1) / PAGE : 0;
      acc += (long long)Hkv * (pages + wch * __popc(window_chunk_mask(L, H)));
    }
    pre[B] = acc;
  }
  __syncthreads();
  Balanced bl;
  bl.W = pre[B];
  bl.n = (int)(bl.W < grid ? bl.W : grid);
  bl.wch = wch;
  return bl;
}

__host__ __device__ __forceinline__ long long balanced_lo(const Balanced& bl, int i) {
  return (long long)i * bl.W / bl.n;
}

// The CTA whose range holds position x (0 <= x < W).
__host__ __device__ __forceinline__ int balanced_owner(const Balanced& bl, long long x) {
  return (int)(((x + 1) * bl.n + bl.W - 1) / bl.W - 1);
}

// Largest b with pre[b] <= x (pre non-decreasing, pre[0] = 0 <= x < pre[B]).
__device__ __forceinline__ int balanced_request(const long long* pre, int B, long long x) {
  int lo = 0, hi = B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (pre[mid] <= x) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// ------------------------------------------------------------- launchers
// Optional per-kernel event recording (see oscar_profile_enable).
struct Profiler;
void prof_begin(Profiler* p, int kernel_id, cudaStream_t st);
void prof_end(Profiler* p, int kernel_id, cudaStream_t st);

struct DecodeArgs {
  CacheView cv;
  const __nv_bfloat16* q;  // [B][Hq][128]
  __nv_bfloat16* out;      // [B][Hq][128]
  float* lse;              // [B][Hq] or null
  float* qrot;             // scratch [B][Hq][128] rotated queries (fp32)
  uint8_t* qpack;          // scratch [B][Hq] packed query records
  float* part;             // scratch partials
  int* counter;            // scratch work counter
  int B;
  int target_items;
  int resident;  // resident decode CTAs for automatic item sizing, 0: fixed items per CTA
  int impl;  // decode kernel variant: 0 tensor-core one page per warp, 1 CUDA-core, 3 tensor-core
             // with page pairs, 4 tensor-core with a Lloyd-Max codebook, 5 tcgen05 with tensor memory
  int bf16_history;
  int merge_hpc;  // query heads per merge CTA (divides G)
  int wait_polls; // budget of each page's first wait in decode_kernel (OSCAR_OPT_WAIT_POLLS)
  // Decode step (step_kernel then decode_kernel): the step kernel writes the
  // lengths its append will leave, pred[0..B) seq, pred[B..2B) hist and
  // pred[2B..3B) the history length before the append, and releases the
  // decode kernel at once; the decode kernel schedules from them and copies
  // the page that receives the demoted token only after its wait.
  int step_pred;
  int32_t* pred;  // scratch [3][B]
  int balanced;   // work partition: 0 item list, 1 balanced (the tensor-memory kernel's always),
                  // 2 decided on the device from the lengths (decode grid in bal_grid)
  int bal_grid;
  int bal_wch;
  LayerRot rot;
};

// Per (request, query head) record of the packed query (QPACK_BYTES):
//   half  qb[128]   q'_c * 2^-sigma * 2^(8 - E(c)), the QK^T B operand
//   float alpha     2^sigma * log2(e) / (256 sqrt(d))
//   float qsum[4]   sum of qb over channels 32k .. 32k + 31
//   float psum[4]   sum of q' over channels 32k .. 32k + 31
// A group of g channels takes its logit offset -1024 * alpha * (sum of qb) and
// its zero-point weight (sum of q') * log2(e) / sqrt(d) from g / 32 quarters.
constexpr int QPACK_ALPHA = 256, QPACK_QSUM = 260, QPACK_PSUM = 276;
// With a Lloyd-Max codebook (decode variant 4) the record is QPACK_CB_BYTES:
//   half  qa[128]   q'_c * 2^-sigma * 2^(8 - E(c)) * alpha_K   (low code bit)
//   half  qb[128]   the same times beta_half_K                  (high code bit)
//   float alpha, float qsum[4] (sums of qa + qb), float psum[4] as above.
constexpr int QPACK_CB_QB = 256, QPACK_CB_ALPHA = 512, QPACK_CB_QSUM = 516, QPACK_CB_PSUM = 532;

// Bulk L2 prefetch of `bytes` (a multiple of 16) at a 16-byte aligned address.
__device__ __forceinline__ void bulk_prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;\n" ::"l"(p), "r"(bytes) : "memory");
}

// L2 prefetch of pages the decode kernel's CTAs copy first, issued by the
// query kernel before its wait (so during the previous kernel's tail).  With
// the item list, the CTA that runs item j of (b, kvh) first copies pages
// jS .. jS + 7 (two per warp); quarter cq of (b, kvh)'s query work prefetches
// jS .. jS + 3 (each warp's first page) of the items j = cq (mod 4) that a
// CTA takes first (items below the decode grid; later ones go by the work
// counter).  All eight pages measured slower than four (100K batch 1: decode
// 28.6 against 27.2 us), and than none (27.9 us).  Every thread derives the
// work plan as the decode does, from the lengths as they are now: they may be
// a step old, and nothing depends on the prefetches but timing.  The
// BF16-history decode (the same item list over BF16 page blocks) takes the
// same prefetch; the balanced partition takes it only with fewer than 16
// (request, kv head) segments (below).
__device__ inline void prefetch_first_pages(const DecodeArgs& a, int b, int kvh, int cq, int t) {
  const CacheView& cv = a.cv;
  if (a.balanced == 1) return;
  const int B = a.B, Hkv = cv.Hkv;
  const int32_t* hl = cv.hist_lens;
  int total = 0;
#pragma unroll 1
  for (int i = 0; i < B; ++i) total += (hl[i] + PAGE - 1) / PAGE;
  total *= Hkv;
  const int wave = auto_wave_pages(a.bf16_history);
  if (total <= 0) return;
  const int32_t* row = cv.page_table + (size_t)b * cv.max_pages_per_req;
  const int pages_b = (hl[b] + PAGE - 1) / PAGE;
  auto fetch = [&](int p) {
    if (p < 0 || p >= pages_b || p >= cv.max_pages_per_req) return;
    const int pid = row[p];
    if (pid >= 0 && pid < cv.num_pages)
      bulk_prefetch_l2(cv.pool + (size_t)pid * cv.page_bytes + (size_t)kvh * cv.head_bytes, (uint32_t)cv.head_bytes);
  };
  if (a.balanced == 2 && (long long)total > (long long)wave * a.bal_grid) {
    // the balanced partition with few (request, kv head) segments (the host
    // leaves the choice to the device below 16): segment (b', kvh') weighs its
    // pages plus bal_wch per non-empty window chunk, CTA i starts at
    // floor(i W / n); this quarter takes the CTAs i = cq (mod 4) whose range
    // starts in (b, kvh)'s pages.  (With many segments this derivation, in
    // every query CTA before its wait, cost more than it saved: batch 32 at
    // 8K-32K, 130.9 -> 149.6 us.)
    long long W = 0, seg = 0, wb = 0;
#pragma unroll 1
    for (int i = 0; i < B; ++i) {
      const int H = hl[i], P = H > 0 ? (H + PAGE - 1) / PAGE : 0;
      const long long w = P + (long long)a.bal_wch * __popc(window_chunk_mask(cv.seq_lens[i], H));
      if (i < b) seg += Hkv * w;
      if (i == b) wb = w;
      W += Hkv * w;
    }
    seg += kvh * wb;
    if (W <= 0 || pages_b <= 0) return;
    Balanced bl;
    bl.W = W;
    bl.n = (int)(W < a.bal_grid ? W : a.bal_grid);
    bl.wch = a.bal_wch;
    int i0 = balanced_owner(bl, seg);
    if (balanced_lo(bl, i0) < seg) ++i0;
    const int i1 = balanced_owner(bl, seg + pages_b - 1);
#pragma unroll 1
    for (int e = t;; e += 128) {
      const int i = i0 + cq + 4 * (e >> 2);
      if (i > i1) break;
      fetch((int)(balanced_lo(bl, i) - seg) + (e & 3));
    }
    return;
  }
  int wch = 5, n_win = 0;
  auto pages_per_item = [&](int items) {
    wch = (5LL * B * Hkv * 4 <= items) ? 5 : 1;
    n_win = B * Hkv * wch;
    int th = items - n_win;
    if (th < (items + 1) / 2) th = (items + 1) / 2;
    const int S = (total + th - 1) / th;
    return S < 1 ? 1 : S;
  };
  int S = pages_per_item(a.resident > 0 ? a.resident : a.target_items);
  if (a.resident > 0 && S > wave) {
    S = pages_per_item(a.target_items);
    if (S < AUTO_MIN_PAGES) S = AUTO_MIN_PAGES;
  } else if (a.resident > 0) {
    const int gr = pages_granule(a.impl);
    S = (S + gr - 1) / gr * gr;
  }
#pragma unroll 1
  for (int iter = 0; iter < 32; ++iter) {
    long long n = 0;
#pragma unroll 1
    for (int i = 0; i < B; ++i) n += (long long)Hkv * (((hl[i] + PAGE - 1) / PAGE + S - 1) / S);
    if (n + n_win <= a.target_items || n <= (long long)B * Hkv) break;
    S += S / 8 > 1 ? S / 8 : 1;
  }
  int first = 0;  // the block that runs item 0 of (b, kvh)
#pragma unroll 1
  for (int i = 0; i < b; ++i) first += Hkv * (((hl[i] + PAGE - 1) / PAGE + S - 1) / S);
  const int nb = (pages_b + S - 1) / S;
  first += kvh * nb + ((long long)(WIN_BYTES_PER_HEAD / wch) > (long long)S * cv.head_bytes ? n_win : 0);
#pragma unroll 1
  for (int e = t;; e += 128) {
    const int j = cq + 4 * (e >> 2);
    if (j >= nb || first + j >= a.bal_grid) break;
    fetch(j * S + (e & 3));
  }
}

struct PrepSmem {
  float xs[MAX_G][D];
  float part[4][MAX_G][32];
  float nrm[MAX_G];
};

// Channels 32cq .. 32cq + 31 of q' = q·R_K for the G query heads of
// (request, kv head) bk, by 128 threads (t = thread in the group, its own
// PrepSmem); warp w = t / 32 sums rows 32w .. 32w + 31 of R_K, lane = channel.
// The fp16 prescale sigma comes from |q|, which bounds every |q'_c| (R_K is
// orthogonal), so the four quarters of a head agree on it without talking to
// each other.  The rotation-table loads (written synchronously by
// oscar_set_rotation) go first, then the body waits for earlier stream work;
// with `release` it then lets its dependents launch (the decode kernel reads
// the cache state before its own wait, so it must start only once that work
// is complete), otherwise the caller releases them later.  All threads of
// the block call it (it synchronises the block).
__device__ __forceinline__ void prep_body(const DecodeArgs& a, int bk, int cq, int t, PrepSmem& sm,
                                          bool release) {
  const CacheView& cv = a.cv;
  const int b = bk / cv.Hkv, kvh = bk % cv.Hkv, w = t >> 5, lane = t & 31;
  const int G = cv.G;
  const int c = 32 * cq + lane;
  // R_K, and this CTA's quarter of the merge's R_V fragments into L2
  float r[32];
  if (!a.bf16_history) {
    const float* R = a.rot.R_K + (size_t)kvh * D * D + (size_t)(32 * w) * D + c;
#pragma unroll
    for (int k = 0; k < 32; ++k) r[k] = __ldg(R + k * D);
    const char* rv = (const char*)(a.rot.RV_frag + (size_t)kvh * RV_FRAG_WORDS) + (size_t)(cq * 128 + t) * 128;
    asm volatile("prefetch.global.L2 [%0];\n" ::"l"(rv));
  }
  {
    // The decode kernel's first reads are the lengths and request b's page
    // table row, each a dependent round trip before its first page copy:
    // bring them into L2 now (a hint only; their values are read after the
    // waits that order them).  The row's 128-byte lines are spread over the
    // request's Hkv x 4 CTAs.
    const int per_req = cv.Hkv * 4, me = kvh * 4 + cq;
    if (t == 0 && me == 0) {
      asm volatile("prefetch.global.L2 [%0];\n" ::"l"(cv.hist_lens + b));
      asm volatile("prefetch.global.L2 [%0];\n" ::"l"(cv.seq_lens + b));
    }
    const int lines = (cv.max_pages_per_req + 31) / 32;
    for (int l = me + per_req * t; l < lines; l += per_req * 128)
      asm volatile("prefetch.global.L2 [%0];\n" ::"l"(cv.page_table + (size_t)b * cv.max_pages_per_req + 32 * (size_t)l));
  }
  prefetch_first_pages(a, b, kvh, cq, t);
  pdl_wait();
  if (release) pdl_launch_dependents();
  if (t == 0 && cq == 0 && bk == 0) a.counter[0] = 0;  // history items after the first wave
  if (a.bf16_history) return;
  const __nv_bfloat16* qg = a.q + ((size_t)b * cv.Hq + kvh * G) * D;
  for (int e = t; e < G * D; e += 128) sm.xs[e / D][e % D] = __bfloat162float(qg[e]);
  __syncthreads();
  for (int n = w; n < G; n += 4) {
    float sq = 0.f;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float v = sm.xs[n][lane + 32 * k];
      sq = fmaf(v, v, sq);
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, o);
    if (lane == 0) sm.nrm[n] = sqrtf(sq);
  }
#pragma unroll
  for (int n = 0; n < MAX_G; ++n) {
    if (n < G) {
      float acc = 0.f;
#pragma unroll
      for (int k = 0; k < 32; ++k) acc = fmaf(sm.xs[n][32 * w + k], r[k], acc);
      sm.part[w][n][lane] = acc;
    }
  }
  __syncthreads();
  const int i = 2 * ((c >> 4) & 3) + ((c >> 3) & 1);  // bit pair holding channel c in QK
  const float f = (float)(1 << (8 - code_exp_rt(i)));
  for (int n = w; n < G; n += 4) {
    const float y = (sm.part[0][n][lane] + sm.part[1][n][lane]) + (sm.part[2][n][lane] + sm.part[3][n][lane]);
    const size_t row = (size_t)b * cv.Hq + kvh * G + n;
    a.qrot[row * D + c] = y;
    // power-of-two prescale so that |q'| * 16 stays below 2^14 in fp16
    const float am = sm.nrm[n];
    // sig = frexp exponent of |q| less 10, from the exponent bits (|q| is a
    // normal float in practice; the clamp keeps 2^-sig a normal float)
    const int sig = am > 0.f ? max(-100, min(100, (int)((__float_as_uint(am) >> 23) & 0xffu) - 136)) : 0;
    const float yq = y * pow2i(-sig) * f;
    const bool cbrec = a.impl == 4;
    uint8_t* rec = a.qpack + row * (cbrec ? QPACK_CB_BYTES : QPACK_BYTES);
    float bs, ps = y;
    if (!cbrec) {
      const __half hb = __float2half_rn(yq);
      ((__half*)rec)[c] = hb;
      bs = __half2float(hb);
    } else {
      const float* cbk = a.rot.cb + (size_t)kvh * CB_WORDS;
      const __half ha = __float2half_rn(yq * __ldg(cbk + CB_ALPHA));
      const __half hb = __float2half_rn(yq * __ldg(cbk + CB_BETA_HALF));
      ((__half*)rec)[c] = ha;
      ((__half*)(rec + QPACK_CB_QB))[c] = hb;
      bs = __half2float(ha) + __half2float(hb);
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      bs += __shfl_xor_sync(0xffffffffu, bs, o);
      ps += __shfl_xor_sync(0xffffffffu, ps, o);
    }
    if (lane == 0) {
      ((float*)(rec + (cbrec ? QPACK_CB_QSUM : QPACK_QSUM)))[cq] = bs;
      ((float*)(rec + (cbrec ? QPACK_CB_PSUM : QPACK_PSUM)))[cq] = ps;
      if (cq == 0)
        *(float*)(rec + (cbrec ? QPACK_CB_ALPHA : QPACK_ALPHA)) = pow2i(sig) * LOG2E * INV_SQRT_D * (1.f / 256.f);
    }
  }
}

cudaError_t launch_decode(const DecodeArgs& a, int grid, cudaStream_t st, Profiler* prof);
// The tensor-memory decode kernel (impl 5, oscar_decode_tc.cu): grid a.bal_grid, balanced partition.
cudaError_t launch_decode_tc(const DecodeArgs& a, cudaStream_t st);
int decode_tc_smem_bytes(int head_bytes, int B);
int decode_tc_window_weight();
// The decode kernel and the merge only (the caller ran the packed query).
cudaError_t launch_decode_after_prep(const DecodeArgs& a, int grid, cudaStream_t st, Profiler* prof);
int decode_ctas_per_sm(const DecodeArgs& a);  // resident CTAs per SM of the decode kernel (0: error)

// Decode scratch: [work counter][predicted lengths][q' fp32][packed q][partials]
struct ScratchLayout {
  size_t off_counter, off_pred, off_qrot, off_qpack, off_part, total;
};
ScratchLayout scratch_layout(int B, int Hq, int Hkv, int G, int max_target_items);
size_t decode_scratch_bytes(int B, int Hq, int Hkv, int G, int max_target_items);

// ----------------------------------------------------------------- prefill
// Chunked prefill over the cache: T new tokens of a request attend to its
// sink, INT2 history and recent window and causally to each other.
constexpr int PF_ROWS = 128;       // query rows (token x head of one kv head) per attention CTA
constexpr int PF_MAX_T = 64;       // chunk tokens per call
constexpr int PF_MAX_SPLITS = 64;  // history splits per row tile

struct PrefillArgs {
  CacheView cv;
  const __nv_bfloat16* q;  // [B][T][Hq][128]
  const __nv_bfloat16* k;  // [B][T][Hkv][128]
  const __nv_bfloat16* v;  // [B][T][Hkv][128]
  __nv_bfloat16* out;      // [B][T][Hq][128]
  float* lse;              // [B][T][Hq] or null
  __half* qh;              // scratch [2][B*Hkv][RT*128][128]: q·R_K, q (both * 2^-sigma)
  float* alpha;            // scratch [B*Hkv][RT*128]: 2^sigma * log2(e) / sqrt(d)
  float* part;             // scratch [B*Hkv*RT][NS+1][128][PART_STRIDE]
  int B, T, RT, NS;
  int impl;  // an oscar_prefill_impl value
  int codebook;  // the layer has a Lloyd-Max codebook (mma.sync kernel only)
  LayerRot rot;
};

struct PrefillScratch {
  size_t off_qh, off_alpha, off_part, total;
};
PrefillScratch prefill_scratch_layout(int B, int Hkv, int G, int T, int NS);
int prefill_max_splits(int B, int Hkv, int G, int T);  // NS bound the scratch is sized for
cudaError_t prefill_ctas_per_sm(int* n, int impl);        // resident attention CTAs per SM
cudaError_t launch_prefill(const PrefillArgs& a, cudaStream_t st, Profiler* prof);

// ------------------------------------------------------------- calibration
// Offline: covariances, eigenbases and clip errors of one (layer, kv head).
struct CalibScratch {
  size_t off_c, off_cf, off_err, off_clips, off_y, off_kr, off_vr, off_e, total;
};
CalibScratch calib_scratch_layout(int G, int N, int M);
// Unnormalised sums into scratch: C_Q = Σ qᵀq over the G·N rows of Q, then
// C_S = Σ_h (S_h V)ᵀ(S_h V) (fp64 [2][128][128] at off_c).
cudaError_t calib_covariances(const __nv_bfloat16* Q, const __nv_bfloat16* K, const __nv_bfloat16* V, int G, int N,
                              uint8_t* scratch, cudaStream_t st);
// Eigenvectors of the symmetric fp64 device matrix dC (column i of the
// column-major result = eigenvector of the i-th smallest eigenvalue), copied to
// host memory; synchronises st.  OSCAR_ERR_UNSUPPORTED when cuSOLVER is absent.
oscar_status calib_eigh(const double* dC, double* evec_host, cudaStream_t st, int* cuda_err);  // process-wide solver state
// Key and value clip errors of M candidate ratios into scratch (fp64 [2][M] at off_err).
// cb_k, cb_v: the head's codebook records (device), applied by the quantiser.
cudaError_t calib_clip_errors(const float* R_K, const float* R_V, const __nv_bfloat16* Q, const __nv_bfloat16* K,
                              const __nv_bfloat16* V, int G, int N, int g, const float* clips_host, int M,
                              const float* cb_k, const float* cb_v, uint8_t* scratch, cudaStream_t st);
// Lloyd-Max codebook of one (kv head, K or V) from N calibration rows X
// rotated by R: folded values into scratch, then the two-level iteration.
// Scratch: codebook_scratch_bytes(N).  ab_host receives (a, b) as doubles and
// updates_host the number of centroid updates; synchronises st.
size_t codebook_scratch_bytes(int N);
cudaError_t calib_fit_codebook(const float* R, const __nv_bfloat16* X, int N, int g, float clip, int max_iters,
                               uint8_t* scratch, double* ab_host, int* updates_host, cudaStream_t st);

cudaError_t launch_append(const CacheView& cv, const LayerRot& rot, const __nv_bfloat16* k,
                          const __nv_bfloat16* v, int B, int do_append, int* req_counter,
                          cudaStream_t st, Profiler* prof);
// One decode step's first kernel: the append (as launch_append) and the packed
// query (as prep_kernel) in one grid.
cudaError_t launch_step(const CacheView& cv, const LayerRot& rot, const __nv_bfloat16* k,
                        const __nv_bfloat16* v, int B, int* req_counter, const DecodeArgs& a,
                        cudaStream_t st, Profiler* prof);
// One token per request into a BF16-history cache (cv over the BF16 pool).
cudaError_t launch_append_bf16(const CacheView& cv, const __nv_bfloat16* k, const __nv_bfloat16* v, int B,
                               cudaStream_t st, Profiler* prof);
cudaError_t launch_import(const CacheView& cv, const LayerRot& rot, const __nv_bfloat16* K,
                          const __nv_bfloat16* V, int B, int n, int bf16_history,
                          cudaStream_t st, Profiler* prof);
cudaError_t launch_quantize_hook(const float* x, int n, int g, float clip, int which, float thr_lo,
                                 float thr_hi, uint8_t* codes, __half2* sz, cudaStream_t st);
cudaError_t launch_debug_rotate(const float* R, const __nv_bfloat16* x, float* y, int n,
                                cudaStream_t st);

}  // namespace oscar
