// Host side of the liboscar C ABI: argument checks, context, rotation tables
// and kernel launches.  See include/oscar.h for the contract of each call.
#include <math.h>
#include <cmath>
#include <stdlib.h>
#include <string.h>

#include <new>
#include <mutex>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "oscar_internal.cuh"

using namespace oscar;

namespace oscar {
// Event pairs recorded around kernel launches while profiling is on.
struct Profiler {
  bool on = false;
  std::vector<cudaEvent_t> pool;  // created lazily, reused
  std::vector<int> kid;           // kernel id per recorded pair
  size_t used = 0;                // events in use (2 per pair)
  cudaEvent_t pending = nullptr;
};

void prof_begin(Profiler* p, int, cudaStream_t st) {
  if (!p || !p->on) return;
  if (p->used + 2 > p->pool.size()) {
    if (p->pool.size() >= 2 * 65536) return;
    cudaEvent_t a, b;
    if (cudaEventCreate(&a) != cudaSuccess) return;
    if (cudaEventCreate(&b) != cudaSuccess) {
      cudaEventDestroy(a);
      return;
    }
    p->pool.push_back(a);
    p->pool.push_back(b);
  }
  p->pending = p->pool[p->used];
  cudaEventRecord(p->pending, st);
}

void prof_end(Profiler* p, int kernel_id, cudaStream_t st) {
  if (!p || !p->on || !p->pending) return;
  cudaEventRecord(p->pool[p->used + 1], st);
  p->kid.push_back(kernel_id);
  p->used += 2;
  p->pending = nullptr;
}
}  // namespace oscar

struct oscar_ctx {
  oscar_config cfg;
  int device = 0;
  int num_sms = 0;
  int G = 0, NG = 0;
  float* d_rot = nullptr;  // [layers][4][Hkv][128 * 128 words]: R_K, R_V, R_V fragments, R_V^T
  float* d_clip = nullptr;  // [layers][2][Hkv]
  float* d_cb = nullptr;    // [layers][2][Hkv][CB_WORDS] codebook records (uniform by default)
  std::vector<int> mode;
  std::vector<int> has_cb;        // [layers] a non-uniform codebook is set: decode variant 4
  std::vector<float> clip_host;   // [layers][2][Hkv] copy of d_clip
  int* d_err = nullptr;
  int* d_req_counter = nullptr;  // [max_batch]
  int impl = 0;
  int ctas_per_sm = 4;
  int items_per_cta = 0;  // 0: automatic (make_sched)
  int prefill_impl = OSCAR_PREFILL_TCGEN05;
  int wait_polls = WAIT_POLLS;
  int partition = 0;  // OSCAR_OPT_DECODE_PARTITION
  Profiler prof;
};

namespace {

constexpr int VERSION = 10000;

// An NVTX range named after the ABI call, for timeline tools (a no-op unless
// a tool is attached; NVTX 3 is header-only).
struct CallRange {
  explicit CallRange(const char* name) { nvtxRangePushA(name); }
  ~CallRange() { nvtxRangePop(); }
  CallRange(const CallRange&) = delete;
  CallRange& operator=(const CallRange&) = delete;
};

bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

oscar_status check_cfg(const oscar_config* c) {
  if (!c) return OSCAR_ERR_INVALID_ARG;
  if (c->head_dim != D || c->page_size != PAGE || c->sink_tokens != SINK ||
      c->recent_tokens != RECENT)
    return OSCAR_ERR_UNSUPPORTED;
  if (c->group_size != 32 && c->group_size != 64 && c->group_size != 128)
    return OSCAR_ERR_UNSUPPORTED;
  if (c->num_layers < 1 || c->num_q_heads < 1 || c->num_kv_heads < 1 || c->max_batch < 1 ||
      c->max_pages_per_req < 1 || c->num_pages < 1)
    return OSCAR_ERR_INVALID_ARG;
  if (c->num_q_heads % c->num_kv_heads) return OSCAR_ERR_INVALID_ARG;
  const int G = c->num_q_heads / c->num_kv_heads;
  if (G != 1 && G != 2 && G != 4 && G != 8) return OSCAR_ERR_UNSUPPORTED;
  if ((long long)c->max_batch * c->num_q_heads > (1LL << 24)) return OSCAR_ERR_INVALID_ARG;
  if ((long long)c->max_pages_per_req * PAGE > (1LL << 30)) return OSCAR_ERR_INVALID_ARG;
  return OSCAR_OK;
}

size_t scratch_for(const oscar_ctx* ctx, int B, int target) {
  return decode_scratch_bytes(B, ctx->cfg.num_q_heads, ctx->cfg.num_kv_heads, ctx->G, target);
}

// Decode kernel variant: 4 tensor cores with the layer's Lloyd-Max codebook
// (whatever the option); 1 CUDA-core INT2; 3 tensor cores, pages in pairs as
// two softmax streams per tile (needs G <= 4); 0 tensor cores, one page at a
// time.  layer < 0: the variant without a codebook.
int kernel_impl(const oscar_ctx* ctx, int layer = -1) {
  if (layer >= 0 && ctx->has_cb[layer]) return 4;
  if (ctx->impl == OSCAR_DECODE_TCGEN05) return 5;
  if (ctx->impl == OSCAR_DECODE_CUDA_CORE) return 1;
  if (ctx->impl == OSCAR_DECODE_TENSOR_SINGLE || ctx->G > 4) return 0;
  return 3;
}

// Persistent decode CTAs per SM: the option, capped by what the kernel variant
// for this call can keep resident.
int decode_ctas(const oscar_ctx* ctx, int batch, bool bf16_history, int layer = -1) {
  DecodeArgs a = {};
  a.cv.head_bytes = bf16_history ? BF16_HEAD_BYTES : int2_head_bytes(ctx->cfg.group_size);
  a.cv.NG = ctx->NG;
  a.cv.G = ctx->G;
  a.B = batch;
  a.impl = bf16_history ? 0 : kernel_impl(ctx, layer);
  a.bf16_history = bf16_history ? 1 : 0;
  int occ = decode_ctas_per_sm(a);
  if (occ < 1) occ = 1;
  return ctx->ctas_per_sm < occ ? ctx->ctas_per_sm : occ;
}

// decode_kernel's work partition (DecodeArgs::balanced): 0 the item list, 1
// balanced, 2 decided on the device (balanced once the item list would give
// a CTA more than a wave's worth of pages).  Automatic: balanced from 16
// (request, kv head) segments on; below that the device decides.  With few
// segments the balanced ranges hand every window chunk of a kv head to the
// CTA or two at the head's end, where the item list spreads them over
// distinct CTAs (batch 1 at 100K: 27.9 us with items, 33.5 balanced); from
// two requests on the balanced ranges measured faster at every batched shape
// tried (batch 2 to 128, 2K to 131K tokens).
int decode_partition(const oscar_ctx* ctx, int batch) {
  if (ctx->partition == 1) return 0;
  if (ctx->partition == 2) return 1;
  return batch * ctx->cfg.num_kv_heads >= 16 ? 1 : 2;
}

// The item list's size bound (make_sched's target).
int list_items(const oscar_ctx* ctx, int batch, bool bf16_history, int layer = -1) {
  const int per = ctx->items_per_cta ? ctx->items_per_cta : AUTO_ITEMS_PER_CTA;
  int t = ctx->num_sms * decode_ctas(ctx, batch, bf16_history, layer) * per;
  if (t > MAX_TARGET_ITEMS) t = MAX_TARGET_ITEMS;
  if (t < 1) t = 1;
  return t;
}

// Partial records the decode may write, less the 2 B Hkv the scratch layout
// adds.  A balanced partition (the tensor-memory kernel's always) writes one
// history record per (CTA, segment) pair and five window records per
// segment: CTAs + 6 B Hkv.
int target_items(const oscar_ctx* ctx, int batch, bool bf16_history, int layer = -1) {
  if (!bf16_history && kernel_impl(ctx, layer) == 5) return ctx->num_sms + 4 * batch * ctx->cfg.num_kv_heads;
  const int t = list_items(ctx, batch, bf16_history, layer);
  const int ctas = ctx->num_sms * decode_ctas(ctx, batch, bf16_history, layer);
  const int tb = ctas + 4 * batch * ctx->cfg.num_kv_heads;
  const int part = decode_partition(ctx, batch);
  if (part == 1) return tb;
  if (part == 2 && tb > t) return tb;
  return t;
}

bool cache_ok(const oscar_cache* c, bool need_pool) {
  if (!c) return false;
  if (need_pool && (!c->pool || !c->page_table || !aligned(c->pool, 256))) return false;
  if (!c->sink_k || !c->sink_v || !c->ring_k || !c->ring_v || !c->seq_lens || !c->hist_lens)
    return false;
  return aligned(c->sink_k, 16) && aligned(c->sink_v, 16) && aligned(c->ring_k, 16) &&
         aligned(c->ring_v, 16) && aligned(c->seq_lens, 4) && aligned(c->hist_lens, 4);
}

CacheView make_view(const oscar_ctx* ctx, const oscar_cache* c, bool bf16_history) {
  CacheView v;
  v.pool = (uint8_t*)c->pool;
  v.page_table = c->page_table;
  v.sink_k = (__nv_bfloat16*)c->sink_k;
  v.sink_v = (__nv_bfloat16*)c->sink_v;
  v.ring_k = (__nv_bfloat16*)c->ring_k;
  v.ring_v = (__nv_bfloat16*)c->ring_v;
  v.seq_lens = c->seq_lens;
  v.hist_lens = c->hist_lens;
  v.Hq = ctx->cfg.num_q_heads;
  v.Hkv = ctx->cfg.num_kv_heads;
  v.G = ctx->G;
  v.g = ctx->cfg.group_size;
  v.NG = ctx->NG;
  v.max_pages_per_req = ctx->cfg.max_pages_per_req;
  v.num_pages = ctx->cfg.num_pages;
  v.head_bytes = bf16_history ? BF16_HEAD_BYTES : int2_head_bytes(ctx->cfg.group_size);
  v.page_bytes = (long long)v.head_bytes * ctx->cfg.num_kv_heads;
  v.err = ctx->d_err;
  return v;
}

constexpr int ROT_MATS = 4;  // R_K, R_V, R_V fragments, R_V^T per layer
static_assert(RV_FRAG_WORDS == D * D, "R_V fragments fill one matrix slot");

// R = U·H·P_br (OSCAR), H (HADAMARD) or I (NONE) for one head, in fp64, in the
// row-vector convention x' = x·R [News "Together AI 开源 OSCAR…", section
// "OSCAR 的不同之处"].  H is the normalised Sylvester Hadamard of order 128
// applied to each row by the fast transform; (x·P_br)_j = x_bitrev(j).
void compose_rotation(const float* U, int mode, double* R) {
  for (int i = 0; i < D; ++i) {
    double row[D];
    for (int k = 0; k < D; ++k) row[k] = mode == OSCAR_ROT_OSCAR ? (double)U[(size_t)i * D + k] : (i == k);
    if (mode != OSCAR_ROT_NONE) {
      for (int h = 1; h < D; h <<= 1)
        for (int k = 0; k < D; ++k)
          if (!(k & h)) {
            const double a = row[k], b = row[k + h];
            row[k] = a + b;
            row[k + h] = a - b;
          }
      const double sc = 1.0 / sqrt((double)D);
      for (int k = 0; k < D; ++k) row[k] *= sc;
    }
    for (int j = 0; j < D; ++j) {
      int br = 0;
      for (int bit = 0; bit < 7; ++bit) br |= ((j >> bit) & 1) << (6 - bit);
      R[(size_t)i * D + j] = mode == OSCAR_ROT_OSCAR ? row[br] : row[j];
    }
  }
}

uint32_t half_pair(__half lo, __half hi) {
  return (uint32_t)__half_as_ushort(lo) | ((uint32_t)__half_as_ushort(hi) << 16);
}

// A = R (rows: output channel, columns: input channel) as fp16 high / low
// mma fragments (layout of rv_frag_index).
void pack_rv_fragments(const double* R, uint32_t* out) {
  for (int part = 0; part < 2; ++part)
    for (int mt = 0; mt < 8; ++mt)
      for (int ks = 0; ks < 8; ++ks)
        for (int lane = 0; lane < 32; ++lane) {
          const int gid = lane >> 2, tq = lane & 3;
          auto el = [&](int r, int c) {
            const double v = R[(size_t)r * D + c];
            const __half hi = __float2half_rn((float)v);
            if (part == 0) return hi;
            return __float2half_rn((float)(v - (double)__half2float(hi)));
          };
          uint32_t* w = out + rv_frag_index(part, mt, ks, lane);
          const int r0 = 16 * mt + gid, c0 = 16 * ks + 2 * tq;
          w[0] = half_pair(el(r0, c0), el(r0, c0 + 1));
          w[1] = half_pair(el(r0 + 8, c0), el(r0 + 8, c0 + 1));
          w[2] = half_pair(el(r0, c0 + 8), el(r0, c0 + 9));
          w[3] = half_pair(el(r0 + 8, c0 + 8), el(r0 + 8, c0 + 9));
        }
}

// One layer's table (ROT_MATS matrices of Hkv heads) from the eigenbases
// (nullptr outside OSCAR mode: identity): R_K, R_V in fp32, R_V as fp16
// high/low mma fragments, then R_V^T in fp32.
void build_layer_table(const float* U_K, const float* U_V, int mode, int Hkv, std::vector<float>& out) {
  const size_t hm = (size_t)D * D, mat = (size_t)Hkv * hm;
  out.assign(ROT_MATS * mat, 0.f);
  std::vector<double> R(hm);
  for (int h = 0; h < Hkv; ++h) {
    for (int t = 0; t < 2; ++t) {
      const float* U = mode == OSCAR_ROT_OSCAR ? (t == 0 ? U_K : U_V) + h * hm : nullptr;
      compose_rotation(U, mode, R.data());
      float* dst = out.data() + t * mat + h * hm;
      for (size_t e = 0; e < hm; ++e) dst[e] = (float)R[e];
      if (t == 1) {
        pack_rv_fragments(R.data(), (uint32_t*)(out.data() + 2 * mat + h * hm));
        float* rt = out.data() + 3 * mat + h * hm;
        for (int i = 0; i < D; ++i)
          for (int j = 0; j < D; ++j) rt[(size_t)i * D + j] = (float)R[(size_t)j * D + i];
      }
    }
  }
}

// The device record of codebook (a, b): thresholds and decode constants in
// float32, lo/hi = 1.5 -/+ m with m = (a + b)/2.
void codebook_record(float a, float b, float* rec) {
  const float m = (a + b) * 0.5f;  // the halving is exact
  for (int i = 0; i < CB_WORDS; ++i) rec[i] = 0.f;
  rec[CB_A] = a;
  rec[CB_B] = b;
  rec[CB_LO] = 1.5f - m;
  rec[CB_HI] = 1.5f + m;
  rec[CB_C0] = 1.5f - b;
  rec[CB_ALPHA] = b - a;
  rec[CB_BETA_HALF] = m;
}

bool codebook_ok(float a, float b) { return std::isfinite(a) && std::isfinite(b) && a >= 0.f && a < b && b <= 3.f; }

LayerRot layer_rot(const oscar_ctx* ctx, int layer) {
  const size_t mat = (size_t)ctx->cfg.num_kv_heads * D * D;
  LayerRot r;
  r.R_K = ctx->d_rot + (size_t)layer * ROT_MATS * mat;
  r.R_V = r.R_K + mat;
  r.RV_frag = (const uint32_t*)(r.R_V + mat);
  r.RVt = r.R_V + 2 * mat;
  r.clip_k = ctx->d_clip + (size_t)layer * 2 * ctx->cfg.num_kv_heads;
  r.clip_v = r.clip_k + ctx->cfg.num_kv_heads;
  r.cb = ctx->d_cb + (size_t)layer * 2 * ctx->cfg.num_kv_heads * CB_WORDS;
  r.mode = ctx->mode[layer];
  return r;
}

thread_local int g_last_cuda_error = 0;

oscar_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return OSCAR_OK;
  g_last_cuda_error = (int)e;
  (void)cudaGetLastError();  // leave no stale error for the next call
  return OSCAR_ERR_CUDA;
}

// Checks the decode arguments and fills `a` and the grid; OSCAR_OK when there
// is work to launch, OSCAR_ERR_STATE (internal) when batch == 0.
oscar_status decode_args(oscar_ctx* ctx, int layer, const oscar_cache* cache, const void* q, void* out,
                         float* lse, void* scratch, size_t scratch_bytes, int batch, bool bf16_history,
                         DecodeArgs& a, int& grid) {
  if (!ctx || !cache_ok(cache, true) || !q || !out || !scratch) return OSCAR_ERR_INVALID_ARG;
  if (layer < 0 || layer >= ctx->cfg.num_layers) return OSCAR_ERR_INVALID_ARG;
  if (batch < 0 || batch > ctx->cfg.max_batch) return OSCAR_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(out, 16) || !aligned(scratch, 256) ||
      (lse && !aligned(lse, 4)))
    return OSCAR_ERR_INVALID_ARG;
  if (batch == 0) return OSCAR_ERR_STATE;
  const int vlayer = bf16_history ? -1 : layer;  // BF16 history has no codes, so no codebook
  const int target = target_items(ctx, batch, bf16_history, vlayer);
  if (scratch_bytes < scratch_for(ctx, batch, target)) return OSCAR_ERR_INVALID_ARG;
  a.cv = make_view(ctx, cache, bf16_history);
  a.q = (const __nv_bfloat16*)q;
  a.out = (__nv_bfloat16*)out;
  a.lse = lse;
  const ScratchLayout sl =
      scratch_layout(batch, ctx->cfg.num_q_heads, ctx->cfg.num_kv_heads, ctx->G, target);
  uint8_t* sp = (uint8_t*)scratch;
  a.counter = (int*)(sp + sl.off_counter);
  a.pred = (int32_t*)(sp + sl.off_pred);
  a.step_pred = 0;
  a.qrot = (float*)(sp + sl.off_qrot);
  a.qpack = sp + sl.off_qpack;
  a.part = (float*)(sp + sl.off_part);
  a.B = batch;
  a.target_items = list_items(ctx, batch, bf16_history, vlayer);  // make_sched's bound
  a.impl = bf16_history ? 0 : kernel_impl(ctx, vlayer);
  a.bf16_history = bf16_history ? 1 : 0;
  a.rot = layer_rot(ctx, layer);
  // heads per merge CTA: halve while the merge would not cover the SMs
  a.wait_polls = ctx->wait_polls;
  a.merge_hpc = ctx->G;
  while (a.merge_hpc % 2 == 0 && batch * ctx->cfg.num_kv_heads * (ctx->G / a.merge_hpc) < ctx->num_sms)
    a.merge_hpc /= 2;
  a.balanced = 0;
  a.bal_grid = 0;
  a.bal_wch = 0;
  if (a.impl == 5) {
    // one CTA per SM (the kernel holds all 512 tensor-memory columns)
    if (decode_tc_smem_bytes(a.cv.head_bytes, batch) > 227 * 1024) return OSCAR_ERR_UNSUPPORTED;
    a.balanced = 1;
    a.bal_grid = ctx->num_sms;
    a.bal_wch = decode_tc_window_weight();
    grid = ctx->num_sms;
    a.resident = 0;
    return OSCAR_OK;
  }
  grid = ctx->num_sms * decode_ctas(ctx, batch, bf16_history, vlayer);
  a.resident = ctx->items_per_cta == 0 ? grid : 0;
  a.balanced = decode_partition(ctx, batch);
  a.bal_grid = grid;
  a.bal_wch = DEC_WIN_WEIGHT;
  return OSCAR_OK;
}

oscar_status decode_common(oscar_ctx* ctx, int layer, const oscar_cache* cache, const void* q,
                           void* out, float* lse, void* scratch, size_t scratch_bytes, int batch,
                           oscar_stream_t stream, bool bf16_history) {
  DecodeArgs a;
  int grid = 0;
  const oscar_status s =
      decode_args(ctx, layer, cache, q, out, lse, scratch, scratch_bytes, batch, bf16_history, a, grid);
  if (s == OSCAR_ERR_STATE) return OSCAR_OK;  // batch == 0: nothing to do
  if (s != OSCAR_OK) return s;
  return cuda_status(launch_decode(a, grid, (cudaStream_t)stream, &ctx->prof));
}

}  // namespace


// ----------------------------------------------- decode without allocation
// The working memory of oscar_decode_noalloc: one buffer per device that the
// library holds for the life of the process.  In host code the symbol is only
// a stand-in; its device address is looked up once per device.
namespace {
static __device__ __align__(256) uint8_t g_noalloc_scratch[OSCAR_NOALLOC_SCRATCH_BYTES];
constexpr int NOALLOC_MAX_DEVICES = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[NOALLOC_MAX_DEVICES] = {};

// The buffer of the context's device.  The address is looked up with that
// device current, so the call is refused when another device is current: the
// lookup would give the other device's copy of the buffer.
oscar_status noalloc_scratch(const oscar_ctx* ctx, void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return cuda_status(cudaErrorInvalidDevice);
  if (dev != ctx->device) return OSCAR_ERR_INVALID_ARG;
  if (dev < 0 || dev >= NOALLOC_MAX_DEVICES) return OSCAR_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p) return cuda_status(e != cudaSuccess ? e : cudaErrorInvalidSymbol);
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return OSCAR_OK;
}
}  // namespace

extern "C" {

int oscar_version(void) { return VERSION; }

const char* oscar_status_string(int s) {
  switch (s) {
    case OSCAR_OK: return "ok";
    case OSCAR_ERR_INVALID_ARG: return "invalid argument";
    case OSCAR_ERR_UNSUPPORTED: return "unsupported configuration";
    case OSCAR_ERR_NO_PAGE: return "page-table entry is -1";
    case OSCAR_ERR_RANGE: return "page id, length or scale out of range";
    case OSCAR_ERR_TIMEOUT: return "bounded device wait ran out";
    case OSCAR_ERR_CUDA: return "CUDA runtime error";
    case OSCAR_ERR_STATE: return "cache state does not allow the call";
    case OSCAR_ERR_TOO_LARGE: return "request needs more than the built-in no-allocation scratch";
    default: return "unknown status";
  }
}

oscar_status oscar_layout(const oscar_config* cfg, oscar_layout_info* out) {
  const oscar_status s = check_cfg(cfg);
  if (s != OSCAR_OK) return s;
  if (!out) return OSCAR_ERR_INVALID_ARG;
  const int g = cfg->group_size;
  const int G = cfg->num_q_heads / cfg->num_kv_heads;
  out->int2_head_bytes = (size_t)int2_head_bytes(g);
  out->int2_page_bytes = out->int2_head_bytes * cfg->num_kv_heads;
  out->off_k_codes = 0;
  out->off_v_codes = 2048;
  out->off_k_sz = (size_t)off_k_sz();
  out->off_v_sz = (size_t)off_v_sz(g);
  out->bf16_head_bytes = BF16_HEAD_BYTES;
  out->bf16_page_bytes = (size_t)BF16_HEAD_BYTES * cfg->num_kv_heads;
  out->sink_bytes = (size_t)cfg->max_batch * cfg->num_kv_heads * SINK * D * 2;
  out->ring_bytes = (size_t)cfg->max_batch * cfg->num_kv_heads * RECENT * D * 2;
  // enough partial records for every decode kernel: the item list of the
  // mma.sync kernels (at most MAX_TARGET_ITEMS) and the tensor-memory
  // kernel's (one per SM, at most MAX_TARGET_ITEMS SMs, plus 4 B Hkv)
  out->decode_scratch_bytes = decode_scratch_bytes(cfg->max_batch, cfg->num_q_heads, cfg->num_kv_heads, G,
                                                   MAX_TARGET_ITEMS + 4 * cfg->max_batch * cfg->num_kv_heads);
  // the split count (and so the partials) is not monotone in the batch: take the largest
  size_t pf = 0;
  for (int b = 1; b <= cfg->max_batch; ++b) {
    const int ns = prefill_max_splits(b, cfg->num_kv_heads, G, PF_MAX_T);
    const size_t t = prefill_scratch_layout(b, cfg->num_kv_heads, G, PF_MAX_T, ns).total;
    if (t > pf) pf = t;
  }
  out->prefill_scratch_bytes = pf;
  return OSCAR_OK;
}

oscar_status oscar_create(const oscar_config* cfg, oscar_ctx** out) {
  const CallRange nvtx_range("oscar_create");
  if (!out) return OSCAR_ERR_INVALID_ARG;
  *out = nullptr;
  const oscar_status s = check_cfg(cfg);
  if (s != OSCAR_OK) return s;
  oscar_ctx* ctx = new (std::nothrow) oscar_ctx();
  if (!ctx) return OSCAR_ERR_INVALID_ARG;
  ctx->cfg = *cfg;
  ctx->G = cfg->num_q_heads / cfg->num_kv_heads;
  ctx->NG = D / cfg->group_size;
  ctx->mode.assign(cfg->num_layers, (int)OSCAR_ROT_NONE);
  ctx->has_cb.assign(cfg->num_layers, 0);
  ctx->clip_host.assign((size_t)cfg->num_layers * 2 * cfg->num_kv_heads, 1.f);
  cudaError_t e = cudaGetDevice(&ctx->device);
  if (e == cudaSuccess)
    e = cudaDeviceGetAttribute(&ctx->num_sms, cudaDevAttrMultiProcessorCount, ctx->device);
  const size_t mat = (size_t)cfg->num_kv_heads * D * D;
  const size_t rot_bytes = (size_t)cfg->num_layers * ROT_MATS * mat * sizeof(float);
  const size_t clip_bytes = (size_t)cfg->num_layers * 2 * cfg->num_kv_heads * sizeof(float);
  if (e == cudaSuccess) e = cudaMalloc((void**)&ctx->d_rot, rot_bytes);
  if (e == cudaSuccess) e = cudaMalloc((void**)&ctx->d_clip, clip_bytes);
  const size_t cb_floats = (size_t)cfg->num_layers * 2 * cfg->num_kv_heads * CB_WORDS;
  if (e == cudaSuccess) e = cudaMalloc((void**)&ctx->d_cb, cb_floats * sizeof(float));
  if (e == cudaSuccess) e = cudaMalloc((void**)&ctx->d_err, sizeof(int));
  if (e == cudaSuccess) e = cudaMalloc((void**)&ctx->d_req_counter, sizeof(int) * cfg->max_batch);
  if (e == cudaSuccess) e = cudaMemset(ctx->d_err, 0, sizeof(int));
  if (e == cudaSuccess) e = cudaMemset(ctx->d_req_counter, 0, sizeof(int) * cfg->max_batch);
  if (e == cudaSuccess) {
    // identity rotation and clip 1.0 until oscar_set_rotation is called
    std::vector<float> eye;
    build_layer_table(nullptr, nullptr, OSCAR_ROT_NONE, cfg->num_kv_heads, eye);
    for (int l = 0; l < cfg->num_layers && e == cudaSuccess; ++l)
      e = cudaMemcpy(ctx->d_rot + (size_t)l * ROT_MATS * mat, eye.data(), ROT_MATS * mat * sizeof(float),
                     cudaMemcpyHostToDevice);
    std::vector<float> ones((size_t)cfg->num_layers * 2 * cfg->num_kv_heads, 1.f);
    if (e == cudaSuccess)
      e = cudaMemcpy(ctx->d_clip, ones.data(), clip_bytes, cudaMemcpyHostToDevice);
    std::vector<float> cb(cb_floats);
    for (size_t i = 0; i < cb_floats; i += CB_WORDS) codebook_record(0.5f, 1.5f, &cb[i]);
    if (e == cudaSuccess)
      e = cudaMemcpy(ctx->d_cb, cb.data(), cb_floats * sizeof(float), cudaMemcpyHostToDevice);
  }
  if (e != cudaSuccess) {
    oscar_destroy(ctx);
    return OSCAR_ERR_CUDA;
  }
  *out = ctx;
  return OSCAR_OK;
}

oscar_status oscar_destroy(oscar_ctx* ctx) {
  const CallRange nvtx_range("oscar_destroy");
  if (!ctx) return OSCAR_ERR_INVALID_ARG;
  cudaDeviceSynchronize();
  if (ctx->d_rot) cudaFree(ctx->d_rot);
  if (ctx->d_clip) cudaFree(ctx->d_clip);
  if (ctx->d_cb) cudaFree(ctx->d_cb);
  if (ctx->d_err) cudaFree(ctx->d_err);
  if (ctx->d_req_counter) cudaFree(ctx->d_req_counter);
  for (cudaEvent_t e : ctx->prof.pool) cudaEventDestroy(e);
  delete ctx;
  return OSCAR_OK;
}

oscar_status oscar_set_option(oscar_ctx* ctx, int option, int value) {
  if (!ctx) return OSCAR_ERR_INVALID_ARG;
  switch (option) {
    case OSCAR_OPT_DECODE_IMPL:
      if (value != OSCAR_DECODE_TENSOR && value != OSCAR_DECODE_CUDA_CORE && value != OSCAR_DECODE_TENSOR_SINGLE &&
          value != OSCAR_DECODE_TCGEN05)
        return OSCAR_ERR_INVALID_ARG;
      ctx->impl = value;
      return OSCAR_OK;
    case OSCAR_OPT_CTAS_PER_SM:
      if (value < 1 || value > 4) return OSCAR_ERR_INVALID_ARG;
      ctx->ctas_per_sm = value;
      return OSCAR_OK;
    case OSCAR_OPT_ITEMS_PER_CTA:
      if (value < 0 || value > 8) return OSCAR_ERR_INVALID_ARG;
      ctx->items_per_cta = value;
      return OSCAR_OK;
    case OSCAR_OPT_PREFILL_IMPL:
      if (value != OSCAR_PREFILL_TCGEN05 && value != OSCAR_PREFILL_MMA_SYNC) return OSCAR_ERR_INVALID_ARG;
      ctx->prefill_impl = value;
      return OSCAR_OK;
    case OSCAR_OPT_WAIT_POLLS:
      if (value < 0) return OSCAR_ERR_INVALID_ARG;
      ctx->wait_polls = value;
      return OSCAR_OK;
    case OSCAR_OPT_DECODE_PARTITION:
      if (value < 0 || value > 2) return OSCAR_ERR_INVALID_ARG;
      ctx->partition = value;
      return OSCAR_OK;
    default:
      return OSCAR_ERR_INVALID_ARG;
  }
}

oscar_status oscar_set_rotation(oscar_ctx* ctx, int layer, const float* U_K, const float* U_V,
                                const float* clip_k, const float* clip_v, int rot_mode,
                                oscar_stream_t stream) {
  const CallRange nvtx_range("oscar_set_rotation");
  if (!ctx || layer < 0 || layer >= ctx->cfg.num_layers || !clip_k || !clip_v)
    return OSCAR_ERR_INVALID_ARG;
  if (rot_mode != OSCAR_ROT_OSCAR && rot_mode != OSCAR_ROT_HADAMARD && rot_mode != OSCAR_ROT_NONE)
    return OSCAR_ERR_INVALID_ARG;
  if (rot_mode == OSCAR_ROT_OSCAR && (!U_K || !U_V)) return OSCAR_ERR_INVALID_ARG;
  const int Hkv = ctx->cfg.num_kv_heads;
  for (int h = 0; h < Hkv; ++h)
    if (!(clip_k[h] > 0.f && clip_k[h] <= 1.f) || !(clip_v[h] > 0.f && clip_v[h] <= 1.f))
      return OSCAR_ERR_INVALID_ARG;
  const size_t mat = (size_t)Hkv * D * D;
  std::vector<float> host;
  build_layer_table(U_K, U_V, rot_mode, Hkv, host);
  std::vector<float> clips(2 * Hkv);
  memcpy(clips.data(), clip_k, Hkv * sizeof(float));
  memcpy(clips.data() + Hkv, clip_v, Hkv * sizeof(float));
  cudaStream_t st = (cudaStream_t)stream;
  cudaError_t e = cudaMemcpyAsync(ctx->d_rot + (size_t)layer * ROT_MATS * mat, host.data(),
                                  ROT_MATS * mat * sizeof(float), cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(ctx->d_clip + (size_t)layer * 2 * Hkv, clips.data(), 2 * Hkv * sizeof(float),
                        cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return OSCAR_ERR_CUDA;
  ctx->mode[layer] = rot_mode;
  memcpy(ctx->clip_host.data() + (size_t)layer * 2 * Hkv, clips.data(), 2 * Hkv * sizeof(float));
  return OSCAR_OK;
}

static oscar_status append_common(oscar_ctx* ctx, int layer, const oscar_cache* cache,
                                  const void* k, const void* v, int batch, oscar_stream_t stream,
                                  int do_append) {
  if (!ctx || !cache_ok(cache, true)) return OSCAR_ERR_INVALID_ARG;
  if (layer < 0 || layer >= ctx->cfg.num_layers) return OSCAR_ERR_INVALID_ARG;
  if (batch < 0 || batch > ctx->cfg.max_batch) return OSCAR_ERR_INVALID_ARG;
  if (do_append && (!k || !v || !aligned(k, 16) || !aligned(v, 16))) return OSCAR_ERR_INVALID_ARG;
  if (batch == 0) return OSCAR_OK;
  const CacheView cv = make_view(ctx, cache, false);
  return cuda_status(launch_append(cv, layer_rot(ctx, layer), (const __nv_bfloat16*)k,
                                   (const __nv_bfloat16*)v, batch, do_append, ctx->d_req_counter,
                                   (cudaStream_t)stream, &ctx->prof));
}

oscar_status oscar_append(oscar_ctx* ctx, int layer, const oscar_cache* cache, const void* k_new,
                          const void* v_new, int batch, oscar_stream_t stream) {
  const CallRange nvtx_range("oscar_append");
  return append_common(ctx, layer, cache, k_new, v_new, batch, stream, 1);
}

oscar_status oscar_demote(oscar_ctx* ctx, int layer, const oscar_cache* cache, int batch,
                          oscar_stream_t stream) {
  const CallRange nvtx_range("oscar_demote");
  return append_common(ctx, layer, cache, nullptr, nullptr, batch, stream, 0);
}

static oscar_status import_common(oscar_ctx* ctx, int layer, const oscar_cache* cache,
                                  const void* K, const void* V, int batch, int n,
                                  oscar_stream_t stream, int bf16_history) {
  if (!ctx || !cache_ok(cache, true) || !K || !V) return OSCAR_ERR_INVALID_ARG;
  if (layer < 0 || layer >= ctx->cfg.num_layers) return OSCAR_ERR_INVALID_ARG;
  if (batch < 0 || batch > ctx->cfg.max_batch || n < 0) return OSCAR_ERR_INVALID_ARG;
  if (!aligned(K, 16) || !aligned(V, 16)) return OSCAR_ERR_INVALID_ARG;
  const long long hist = n > SINK + RECENT ? (long long)n - SINK - RECENT : 0;
  if ((hist + PAGE - 1) / PAGE > ctx->cfg.max_pages_per_req) return OSCAR_ERR_INVALID_ARG;
  if (batch == 0 || n == 0) return OSCAR_OK;
  const CacheView cv = make_view(ctx, cache, bf16_history != 0);
  return cuda_status(launch_import(cv, layer_rot(ctx, layer), (const __nv_bfloat16*)K,
                                   (const __nv_bfloat16*)V, batch, n, bf16_history,
                                   (cudaStream_t)stream, &ctx->prof));
}

oscar_status oscar_import_tokens(oscar_ctx* ctx, int layer, const oscar_cache* cache, const void* K,
                                 const void* V, int batch, int n, oscar_stream_t stream) {
  const CallRange nvtx_range("oscar_import_tokens");
  return import_common(ctx, layer, cache, K, V, batch, n, stream, 0);
}

oscar_status oscar_import_bf16_history(oscar_ctx* ctx, const oscar_cache* cache, const void* K,
                                       const void* V, int batch, int n, oscar_stream_t stream) {
  const CallRange nvtx_range("oscar_import_bf16_history");
  return import_common(ctx, 0, cache, K, V, batch, n, stream, 1);
}

oscar_status oscar_append_bf16_history(oscar_ctx* ctx, const oscar_cache* cache, const void* k_new,
                                       const void* v_new, int batch, oscar_stream_t stream) {
  const CallRange nvtx_range("oscar_append_bf16_history");
  if (!ctx || !cache_ok(cache, true) || !k_new || !v_new) return OSCAR_ERR_INVALID_ARG;
  if (batch < 0 || batch > ctx->cfg.max_batch || !aligned(k_new, 16) || !aligned(v_new, 16))
    return OSCAR_ERR_INVALID_ARG;
  if (batch == 0) return OSCAR_OK;
  const CacheView cv = make_view(ctx, cache, true);
  return cuda_status(launch_append_bf16(cv, (const __nv_bfloat16*)k_new, (const __nv_bfloat16*)v_new, batch,
                                        (cudaStream_t)stream, &ctx->prof));
}

oscar_status oscar_decode(oscar_ctx* ctx, int layer, const oscar_cache* cache, const void* q,
                          void* out, float* lse, void* scratch, size_t scratch_bytes, int batch,
                          oscar_stream_t stream) {
  const CallRange nvtx_range("oscar_decode");
  return decode_common(ctx, layer, cache, q, out, lse, scratch, scratch_bytes, batch, stream, false);
}

oscar_status oscar_decode_step(oscar_ctx* ctx, int layer, const oscar_cache* cache,
                               const void* k_new, const void* v_new, const void* q, void* out,
                               float* lse, void* scratch, size_t scratch_bytes, int batch,
                               oscar_stream_t stream) {
  const CallRange nvtx_range("oscar_decode_step");
  if (!k_new || !v_new || !aligned(k_new, 16) || !aligned(v_new, 16)) return OSCAR_ERR_INVALID_ARG;
  DecodeArgs a;
  int grid = 0;
  const oscar_status s =
      decode_args(ctx, layer, cache, q, out, lse, scratch, scratch_bytes, batch, false, a, grid);
  if (s == OSCAR_ERR_STATE) return OSCAR_OK;  // batch == 0: nothing to do
  if (s != OSCAR_OK) return s;
  // the mma.sync decode kernels start on the step kernel's predicted lengths
  a.step_pred = a.impl == 5 ? 0 : 1;
  const cudaStream_t st = (cudaStream_t)stream;
  cudaError_t e = launch_step(a.cv, a.rot, (const __nv_bfloat16*)k_new, (const __nv_bfloat16*)v_new, batch,
                              ctx->d_req_counter, a, st, &ctx->prof);
  if (e == cudaSuccess) e = launch_decode_after_prep(a, grid, st, &ctx->prof);
  return cuda_status(e);
}

oscar_status oscar_prefill(oscar_ctx* ctx, int layer, const oscar_cache* cache, const void* q,
                           const void* k, const void* v, int T, void* out, float* lse,
                           void* scratch, size_t scratch_bytes, int batch, oscar_stream_t stream) {
  const CallRange nvtx_range("oscar_prefill");
  if (!ctx || !cache_ok(cache, true) || !q || !k || !v || !out || !scratch) return OSCAR_ERR_INVALID_ARG;
  if (layer < 0 || layer >= ctx->cfg.num_layers) return OSCAR_ERR_INVALID_ARG;
  if (batch < 0 || batch > ctx->cfg.max_batch || T < 1 || T > PF_MAX_T) return OSCAR_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16) ||
      !aligned(scratch, 256) || (lse && !aligned(lse, 4)))
    return OSCAR_ERR_INVALID_ARG;
  if (batch == 0) return OSCAR_OK;
  // a layer with a Lloyd-Max codebook runs the mma.sync kernel, whose tile
  // fill dequantises codebook levels (the tcgen05 producers do uniform codes)
  const int impl = ctx->has_cb[layer] ? (int)OSCAR_PREFILL_MMA_SYNC : ctx->prefill_impl;
  const int Hkv = ctx->cfg.num_kv_heads, G = ctx->G;
  PrefillArgs a;
  a.RT = (T * G + PF_ROWS - 1) / PF_ROWS;
  const int tiles = batch * Hkv * a.RT;
  int occ = 0;
  const cudaError_t oe = prefill_ctas_per_sm(&occ, impl);
  if (oe != cudaSuccess) return cuda_status(oe);
  if (occ < 1) occ = 1;
  // history splits: the history CTAs fill one wave over the SMs; the light
  // window CTAs (blockIdx.y = NS, launched after every history CTA) take the
  // SMs left over and whatever frees up first, within the scratch bound
  int ns = (ctx->num_sms * occ) / tiles;
  const int cap = prefill_max_splits(batch, Hkv, G, T);
  a.NS = ns < 1 ? 1 : ns > cap ? cap : ns;
  const PrefillScratch L = prefill_scratch_layout(batch, Hkv, G, T, a.NS);
  if (scratch_bytes < L.total) return OSCAR_ERR_INVALID_ARG;
  a.cv = make_view(ctx, cache, false);
  a.q = (const __nv_bfloat16*)q;
  a.k = (const __nv_bfloat16*)k;
  a.v = (const __nv_bfloat16*)v;
  a.out = (__nv_bfloat16*)out;
  a.lse = lse;
  uint8_t* sp = (uint8_t*)scratch;
  a.qh = (__half*)(sp + L.off_qh);
  a.alpha = (float*)(sp + L.off_alpha);
  a.part = (float*)(sp + L.off_part);
  a.B = batch;
  a.T = T;
  a.impl = impl;
  a.codebook = ctx->has_cb[layer];
  a.rot = layer_rot(ctx, layer);
  return cuda_status(launch_prefill(a, (cudaStream_t)stream, &ctx->prof));
}

size_t oscar_calibration_scratch_bytes(int G, int N, int M) {
  if (G < 1 || N < 1 || M < 0) return 0;
  return calib_scratch_layout(G, N, M).total;
}

namespace {
// Column-major eigenvectors of ascending eigenvalues -> row-major U with
// column i = eigenvector of the i-th largest, largest-|.| entry positive.
void order_eigenvectors(const double* evec, float* U) {
  for (int i = 0; i < D; ++i) {
    const double* v = evec + (size_t)(D - 1 - i) * D;
    int arg = 0;
    for (int r = 1; r < D; ++r)
      if (fabs(v[r]) > fabs(v[arg])) arg = r;
    const double sg = v[arg] < 0 ? -1.0 : 1.0;
    for (int r = 0; r < D; ++r) U[(size_t)r * D + i] = (float)(sg * v[r]);
  }
}
}  // namespace

oscar_status oscar_calibrate(oscar_ctx* ctx, const void* Q, const void* K, const void* V, int N, float* U_K,
                             float* U_V, double* C_Q, double* C_S, void* scratch, size_t scratch_bytes,
                             oscar_stream_t stream) {
  const CallRange nvtx_range("oscar_calibrate");
  if (!ctx || !Q || !K || !V || !U_K || !U_V || !scratch || N < 1) return OSCAR_ERR_INVALID_ARG;
  if (!aligned(scratch, 256) || !aligned(Q, 16) || !aligned(K, 16) || !aligned(V, 16)) return OSCAR_ERR_INVALID_ARG;
  const int G = ctx->G;
  const CalibScratch L = calib_scratch_layout(G, N, 0);
  if (scratch_bytes < L.total) return OSCAR_ERR_INVALID_ARG;
  const cudaStream_t st = (cudaStream_t)stream;
  uint8_t* sp = (uint8_t*)scratch;
  cudaError_t e = calib_covariances((const __nv_bfloat16*)Q, (const __nv_bfloat16*)K, (const __nv_bfloat16*)V, G, N,
                                    sp, st);
  if (e != cudaSuccess) return cuda_status(e);
  const double* dC = (const double*)(sp + L.off_c);
  if (C_Q || C_S) {
    std::vector<double> h(2 * D * D);
    e = cudaMemcpyAsync(h.data(), dC, h.size() * sizeof(double), cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_status(e);
    const double inv = 1.0 / ((double)G * N);
    for (int i = 0; i < D * D; ++i) {
      if (C_Q) C_Q[i] = h[i] * inv;
      if (C_S) C_S[i] = h[D * D + i] * inv;
    }
  }
  std::vector<double> evec(D * D);
  for (int t = 0; t < 2; ++t) {
    int ce = 0;
    const oscar_status s = calib_eigh(dC + (size_t)t * D * D, evec.data(), st, &ce);
    if (s == OSCAR_ERR_CUDA && ce) return cuda_status((cudaError_t)ce);
    if (s != OSCAR_OK) return s;
    order_eigenvectors(evec.data(), t == 0 ? U_K : U_V);
  }
  return OSCAR_OK;
}

oscar_status oscar_clip_errors(oscar_ctx* ctx, int layer, int kv_head, const void* Q, const void* K, const void* V,
                               int N, const float* ratios, int M, double* err_k, double* err_v, int* best_k,
                               int* best_v, void* scratch, size_t scratch_bytes, oscar_stream_t stream) {
  const CallRange nvtx_range("oscar_clip_errors");
  if (!ctx || !Q || !K || !V || !ratios || !err_k || !err_v || !scratch || N < 1 || M < 1)
    return OSCAR_ERR_INVALID_ARG;
  if (layer < 0 || layer >= ctx->cfg.num_layers || kv_head < 0 || kv_head >= ctx->cfg.num_kv_heads)
    return OSCAR_ERR_INVALID_ARG;
  if (!aligned(scratch, 256) || !aligned(Q, 16) || !aligned(K, 16) || !aligned(V, 16)) return OSCAR_ERR_INVALID_ARG;
  for (int m = 0; m < M; ++m)
    if (!(ratios[m] > 0.f && ratios[m] <= 1.f)) return OSCAR_ERR_INVALID_ARG;
  const int G = ctx->G;
  const CalibScratch L = calib_scratch_layout(G, N, M);
  if (scratch_bytes < L.total) return OSCAR_ERR_INVALID_ARG;
  const cudaStream_t st = (cudaStream_t)stream;
  const LayerRot r = layer_rot(ctx, layer);
  uint8_t* sp = (uint8_t*)scratch;
  cudaError_t e = calib_clip_errors(r.R_K + (size_t)kv_head * D * D, r.R_V + (size_t)kv_head * D * D,
                                    (const __nv_bfloat16*)Q, (const __nv_bfloat16*)K, (const __nv_bfloat16*)V, G, N,
                                    ctx->cfg.group_size, ratios, M, r.cb + (size_t)kv_head * CB_WORDS,
                                    r.cb + (size_t)(ctx->cfg.num_kv_heads + kv_head) * CB_WORDS, sp, st);
  if (e != cudaSuccess) return cuda_status(e);
  std::vector<double> h(2 * (size_t)M);
  e = cudaMemcpyAsync(h.data(), sp + L.off_err, h.size() * sizeof(double), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_status(e);
  int bk = 0, bv = 0;
  for (int m = 0; m < M; ++m) {
    err_k[m] = h[m];
    err_v[m] = h[M + m];
    if (h[m] < h[bk]) bk = m;
    if (h[M + m] < h[M + bv]) bv = m;
  }
  if (best_k) *best_k = bk;
  if (best_v) *best_v = bv;
  return OSCAR_OK;
}

oscar_status oscar_decode_noalloc(oscar_ctx* ctx, int layer, const oscar_cache* cache,
                                  const void* q, void* out, float* lse, int batch,
                                  oscar_stream_t stream) {
  const CallRange nvtx_range("oscar_decode_noalloc");
  if (!ctx || batch < 0 || batch > ctx->cfg.max_batch) return OSCAR_ERR_INVALID_ARG;
  if (layer < 0 || layer >= ctx->cfg.num_layers) return OSCAR_ERR_INVALID_ARG;
  if (scratch_for(ctx, batch, target_items(ctx, batch, false, layer)) > (size_t)OSCAR_NOALLOC_SCRATCH_BYTES)
    return OSCAR_ERR_TOO_LARGE;
  void* scratch = nullptr;
  const oscar_status st = noalloc_scratch(ctx, &scratch);
  if (st != OSCAR_OK) return st;
  return decode_common(ctx, layer, cache, q, out, lse, scratch, OSCAR_NOALLOC_SCRATCH_BYTES, batch,
                       stream, false);
}

oscar_status oscar_decode_bf16_history(oscar_ctx* ctx, const oscar_cache* cache, const void* q,
                                       void* out, float* lse, void* scratch, size_t scratch_bytes,
                                       int batch, oscar_stream_t stream) {
  const CallRange nvtx_range("oscar_decode_bf16_history");
  return decode_common(ctx, 0, cache, q, out, lse, scratch, scratch_bytes, batch, stream, true);
}

oscar_status oscar_quantize_rotated_f32(const float* x, int n, int group_size, float clip,
                                        int which, uint8_t* codes, void* sz,
                                        oscar_stream_t stream) {
  if (!x || !codes || !sz || n < 0) return OSCAR_ERR_INVALID_ARG;
  if (group_size != 32 && group_size != 64 && group_size != 128) return OSCAR_ERR_UNSUPPORTED;
  if (which != 0 && which != 1) return OSCAR_ERR_INVALID_ARG;
  if (which == 1 && (n % PAGE)) return OSCAR_ERR_INVALID_ARG;
  if (!(clip > 0.f && clip <= 1.f)) return OSCAR_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(codes, 16) || !aligned(sz, 4)) return OSCAR_ERR_INVALID_ARG;
  if (n == 0) return OSCAR_OK;
  return cuda_status(launch_quantize_hook(x, n, group_size, clip, which, 0.5f, 2.5f, codes, (__half2*)sz,
                                          (cudaStream_t)stream));
}

oscar_status oscar_quantize_codebook_f32(const float* x, int n, int group_size, float clip, float a, float b,
                                         int which, uint8_t* codes, void* sz, oscar_stream_t stream) {
  if (!x || !codes || !sz || n < 0) return OSCAR_ERR_INVALID_ARG;
  if (group_size != 32 && group_size != 64 && group_size != 128) return OSCAR_ERR_UNSUPPORTED;
  if (which != 0 && which != 1) return OSCAR_ERR_INVALID_ARG;
  if (which == 1 && (n % PAGE)) return OSCAR_ERR_INVALID_ARG;
  if (!(clip > 0.f && clip <= 1.f) || !codebook_ok(a, b)) return OSCAR_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(codes, 16) || !aligned(sz, 4)) return OSCAR_ERR_INVALID_ARG;
  if (n == 0) return OSCAR_OK;
  float rec[CB_WORDS];
  codebook_record(a, b, rec);
  return cuda_status(launch_quantize_hook(x, n, group_size, clip, which, rec[CB_LO], rec[CB_HI], codes,
                                          (__half2*)sz, (cudaStream_t)stream));
}

oscar_status oscar_set_codebook(oscar_ctx* ctx, int layer, const float* k_ab, const float* v_ab,
                                oscar_stream_t stream) {
  const CallRange nvtx_range("oscar_set_codebook");
  if (!ctx || layer < 0 || layer >= ctx->cfg.num_layers) return OSCAR_ERR_INVALID_ARG;
  const int Hkv = ctx->cfg.num_kv_heads;
  std::vector<float> rec((size_t)2 * Hkv * CB_WORDS);
  bool any = false;
  for (int side = 0; side < 2; ++side) {
    const float* ab = side == 0 ? k_ab : v_ab;
    for (int h = 0; h < Hkv; ++h) {
      const float a = ab ? ab[2 * h] : 0.5f, b = ab ? ab[2 * h + 1] : 1.5f;
      if (!codebook_ok(a, b)) return OSCAR_ERR_INVALID_ARG;
      if (a != 0.5f || b != 1.5f) any = true;
      codebook_record(a, b, &rec[((size_t)side * Hkv + h) * CB_WORDS]);
    }
  }
  const cudaStream_t st = (cudaStream_t)stream;
  cudaError_t e = cudaMemcpyAsync(ctx->d_cb + (size_t)layer * rec.size(), rec.data(), rec.size() * sizeof(float),
                                  cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_status(e);
  ctx->has_cb[layer] = any ? 1 : 0;
  return OSCAR_OK;
}

size_t oscar_codebook_scratch_bytes(int N) {
  if (N < 1 || N > OSCAR_CODEBOOK_MAX_ROWS) return 0;
  return codebook_scratch_bytes(N);
}

oscar_status oscar_fit_codebook(oscar_ctx* ctx, int layer, int kv_head, int which, const void* X, int N,
                                int max_iters, void* scratch, size_t scratch_bytes, float* ab, int* updates,
                                oscar_stream_t stream) {
  const CallRange nvtx_range("oscar_fit_codebook");
  if (!ctx || !X || !scratch || !ab || (which != 0 && which != 1)) return OSCAR_ERR_INVALID_ARG;
  if (layer < 0 || layer >= ctx->cfg.num_layers || kv_head < 0 || kv_head >= ctx->cfg.num_kv_heads)
    return OSCAR_ERR_INVALID_ARG;
  if (N < 1 || N > OSCAR_CODEBOOK_MAX_ROWS || max_iters < 1) return OSCAR_ERR_INVALID_ARG;
  if (!aligned(scratch, 256) || !aligned(X, 16)) return OSCAR_ERR_INVALID_ARG;
  if (scratch_bytes < codebook_scratch_bytes(N)) return OSCAR_ERR_INVALID_ARG;
  const int Hkv = ctx->cfg.num_kv_heads;
  const LayerRot r = layer_rot(ctx, layer);
  const float* R = (which == 0 ? r.R_K : r.R_V) + (size_t)kv_head * D * D;
  const float clip = ctx->clip_host[(size_t)layer * 2 * Hkv + (size_t)which * Hkv + kv_head];
  double h[2];
  int up = 0;
  const cudaError_t e = calib_fit_codebook(R, (const __nv_bfloat16*)X, N, ctx->cfg.group_size, clip, max_iters,
                                           (uint8_t*)scratch, h, &up, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_status(e);
  ab[0] = (float)h[0];
  ab[1] = (float)h[1];
  if (updates) *updates = up;
  return OSCAR_OK;
}

oscar_status oscar_debug_rotate(oscar_ctx* ctx, int layer, int which, int kv_head, const void* x,
                                float* x_rot, int n, oscar_stream_t stream) {
  if (!ctx || !x || !x_rot || n < 0 || (which != 0 && which != 1)) return OSCAR_ERR_INVALID_ARG;
  if (layer < 0 || layer >= ctx->cfg.num_layers) return OSCAR_ERR_INVALID_ARG;
  if (kv_head < 0 || kv_head >= ctx->cfg.num_kv_heads) return OSCAR_ERR_INVALID_ARG;
  if (n == 0) return OSCAR_OK;
  const LayerRot r = layer_rot(ctx, layer);
  const float* R = (which == 0 ? r.R_K : r.R_V) + (size_t)kv_head * D * D;
  return cuda_status(launch_debug_rotate(R, (const __nv_bfloat16*)x, x_rot, n,
                                         (cudaStream_t)stream));
}

oscar_status oscar_check_cache_host(const oscar_config* cfg, const int32_t* seq_lens, const int32_t* hist_lens,
                                    const int32_t* page_table, int batch, int* bad_request) {
  if (bad_request) *bad_request = -1;
  const oscar_status cs = check_cfg(cfg);
  if (cs != OSCAR_OK) return cs;
  if (!seq_lens || !hist_lens || !page_table || batch < 0 || batch > cfg->max_batch) return OSCAR_ERR_INVALID_ARG;
  std::vector<int32_t> owner((size_t)cfg->num_pages, -1);
  for (int b = 0; b < batch; ++b) {
    const long long L = seq_lens[b], H = hist_lens[b];
    oscar_status st = OSCAR_OK;
    const long long lo = L > SINK + RECENT ? L - SINK - RECENT : 0, hi = L > SINK ? L - SINK : 0;
    if (L < 0 || H < lo || H > hi) st = OSCAR_ERR_STATE;
    const long long pages = (H + PAGE - 1) / PAGE;
    if (st == OSCAR_OK && pages > cfg->max_pages_per_req) st = OSCAR_ERR_RANGE;
    for (long long p = 0; st == OSCAR_OK && p < pages; ++p) {
      const int32_t id = page_table[(size_t)b * cfg->max_pages_per_req + p];
      if (id < 0) st = OSCAR_ERR_NO_PAGE;
      else if (id >= cfg->num_pages || owner[id] >= 0) st = OSCAR_ERR_RANGE;
      else owner[id] = b;
    }
    if (st != OSCAR_OK) {
      if (bad_request) *bad_request = b;
      return st;
    }
  }
  return OSCAR_OK;
}

int oscar_last_cuda_error(void) { return g_last_cuda_error; }

oscar_status oscar_get_error(oscar_ctx* ctx, oscar_stream_t stream, int* code) {
  if (!ctx || !code) return OSCAR_ERR_INVALID_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  int h = 0;
  cudaError_t e = cudaMemcpyAsync(&h, ctx->d_err, sizeof(int), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaMemsetAsync(ctx->d_err, 0, sizeof(int), st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return OSCAR_ERR_CUDA;
  *code = h;
  return OSCAR_OK;
}

oscar_status oscar_profile_enable(oscar_ctx* ctx, int enable) {
  if (!ctx) return OSCAR_ERR_INVALID_ARG;
  ctx->prof.on = enable != 0;
  return OSCAR_OK;
}

oscar_status oscar_profile_read(oscar_ctx* ctx, int kernel_id, int* launches, double* total_ms,
                                int reset) {
  if (!ctx || !launches || !total_ms || kernel_id < 0 || kernel_id >= OSCAR_KERNEL_COUNT)
    return OSCAR_ERR_INVALID_ARG;
  Profiler& p = ctx->prof;
  int n = 0;
  double ms = 0.0;
  for (size_t i = 0; i < p.kid.size(); ++i) {
    if (p.kid[i] != kernel_id) continue;
    if (cudaEventSynchronize(p.pool[2 * i + 1]) != cudaSuccess) return cuda_status(cudaErrorUnknown);
    float t = 0.f;
    if (cudaEventElapsedTime(&t, p.pool[2 * i], p.pool[2 * i + 1]) != cudaSuccess)
      return cuda_status(cudaErrorUnknown);
    ms += t;
    ++n;
  }
  *launches = n;
  *total_ms = ms;
  if (reset) {
    p.kid.clear();
    p.used = 0;
  }
  return OSCAR_OK;
}

}  // extern "C"
