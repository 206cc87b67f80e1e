// Offline calibration on the GPU (sm_103a): the rotation bases and the clip
// search of one (layer, kv head) from N calibration tokens.
//
// [News, "OSCAR 的不同之处"]: the key basis is the eigenbasis of the query
// covariance C_Q = (1/N) Σ qᵀq (the logit error of a key perturbation is
// weighted by QᵀQ); the value basis is the eigenbasis of C_S = (1/N) VᵀSᵀSV,
// S the attention scores.  [Blog, "OSCAR把旋转对准attention"]: rotation and
// clipping thresholds are fixed offline per layer and head.
//
//   gram_kernel         C += XᵀX over rows of X (fp32 accumulation per CTA,
//                       fp64 across CTAs)
//   causal_attn_kernel  Y_h = S_h X with S_h = causal softmax(Q_h Kᵀ/√d):
//                       X = V gives the score-weighted values for C_S, X = the
//                       values' quantisation error gives the value clip error
//   quant_err_kernel    rows quantised with the demotion's quantiser at each
//                       candidate ratio; the error x' - x̂' per element
//   key_err_kernel      Σ_n e_n (Q'ᵀQ') e_nᵀ = ||Q' Eᵀ||²_F, the logit error
// The eigen-decomposition is cuSOLVER's dsyevd on the fp64 matrices, opened at
// run time so that the rest of the library does not depend on cuSOLVER.
#include <dlfcn.h>
#include <cusolverDn.h>

#include <algorithm>
#include <mutex>
#include <vector>

#include "oscar_internal.cuh"

namespace oscar {
namespace {

template <typename T>
__device__ __forceinline__ float to_f(T x);
template <>
__device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 x) {
  return __bfloat162float(x);
}
template <>
__device__ __forceinline__ float to_f<float>(float x) {
  return x;
}

constexpr int GRAM_ROWS = 64;  // rows per CTA

// C (fp64 [128][128]) += XᵀX over `rows` rows (row stride 128).  Thread (ti, tj)
// owns the 8x8 output block at (8 ti, 8 tj).
template <typename T>
__global__ void __launch_bounds__(256) gram_kernel(const T* __restrict__ X, int rows, double* C) {
  __shared__ __align__(16) float xs[GRAM_ROWS][D];
  const int tid = threadIdx.x, ti = tid >> 4, tj = tid & 15;
  const int r0 = blockIdx.x * GRAM_ROWS;
  for (int e = tid; e < GRAM_ROWS * D; e += 256) {
    const int r = e / D, c = e % D;
    xs[r][c] = r0 + r < rows ? to_f<T>(X[(size_t)(r0 + r) * D + c]) : 0.f;
  }
  __syncthreads();
  float acc[8][8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;
  for (int r = 0; r < GRAM_ROWS; ++r) {
    const float4 a0 = *(const float4*)&xs[r][8 * ti], a1 = *(const float4*)&xs[r][8 * ti + 4];
    const float4 b0 = *(const float4*)&xs[r][8 * tj], b1 = *(const float4*)&xs[r][8 * tj + 4];
    const float a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
    const float b[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
  }
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) atomicAdd(&C[(8 * ti + i) * D + 8 * tj + j], (double)acc[i][j]);
}

constexpr int ATT_ROWS = 32;  // query rows per CTA (8 warps x 4)
constexpr int ATT_KEYS = 64;  // keys per tile
constexpr int ATT_SMEM = (ATT_ROWS * D + ATT_KEYS * (D + 1) + ATT_KEYS * D + 8 * 4 * ATT_KEYS) * 4;

// Y[h][r] = Σ_{n <= r} softmax_n(q_{h,r}·k_n / √d) x_n for the G heads (grid.y),
// fp32 with an online softmax over key tiles.  With sq, also adds Σ |Y|² to *sq.
template <typename TX>
__global__ void __launch_bounds__(256, 1) causal_attn_kernel(const __nv_bfloat16* __restrict__ Q,
                                                          const __nv_bfloat16* __restrict__ K,
                                                          const TX* __restrict__ X, int N, float* Y,
                                                          double* sq) {
  extern __shared__ __align__(16) float asm_[];
  float* qs = asm_;                         // [32][128]
  float* ks = qs + ATT_ROWS * D;            // [64][129]
  float* xs = ks + ATT_KEYS * (D + 1);      // [64][128]
  float* ps = xs + ATT_KEYS * D;            // [8 warps][4 rows][64]
  const int h = blockIdx.y, r0 = blockIdx.x * ATT_ROWS;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const __nv_bfloat16* Qh = Q + (size_t)h * N * D;
  for (int e = tid; e < ATT_ROWS * D; e += 256) {
    const int r = e / D, c = e % D;
    qs[e] = r0 + r < N ? __bfloat162float(Qh[(size_t)(r0 + r) * D + c]) : 0.f;
  }
  float m[4], l[4], o[4][4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    m[j] = -INFINITY;
    l[j] = 0.f;
#pragma unroll
    for (int k = 0; k < 4; ++k) o[j][k] = 0.f;
  }
  const float scale = rsqrtf((float)D);
  const int last = min(r0 + ATT_ROWS, N) - 1;  // the last key any row of this CTA sees
  for (int t0 = 0; t0 <= last; t0 += ATT_KEYS) {
    __syncthreads();
    for (int e = tid; e < ATT_KEYS * D; e += 256) {
      const int n = e / D, c = e % D;
      const bool in = t0 + n < N;
      ks[n * (D + 1) + c] = in ? __bfloat162float(K[(size_t)(t0 + n) * D + c]) : 0.f;
      xs[n * D + c] = in ? to_f<TX>(X[(size_t)(t0 + n) * D + c]) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int rl = 4 * warp + j, r = r0 + rl;
      float s[2];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int n = lane + 32 * u;
        float acc = 0.f;
#pragma unroll 8
        for (int c = 0; c < D; ++c) acc = fmaf(qs[rl * D + c], ks[n * (D + 1) + c], acc);
        s[u] = (t0 + n <= r && t0 + n < N) ? acc * scale : -INFINITY;
      }
      float mx = fmaxf(s[0], s[1]);
#pragma unroll
      for (int off = 16; off; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      const float mn = fmaxf(m[j], mx);
      const float f = mn == -INFINITY ? 1.f : expf(m[j] - mn);
      const float p0 = mn == -INFINITY ? 0.f : expf(s[0] - mn), p1 = mn == -INFINITY ? 0.f : expf(s[1] - mn);
      float ls = p0 + p1;
#pragma unroll
      for (int off = 16; off; off >>= 1) ls += __shfl_xor_sync(0xffffffffu, ls, off);
      m[j] = mn;
      l[j] = l[j] * f + ls;
#pragma unroll
      for (int k = 0; k < 4; ++k) o[j][k] *= f;
      ps[(warp * 4 + j) * ATT_KEYS + lane] = p0;
      ps[(warp * 4 + j) * ATT_KEYS + lane + 32] = p1;
    }
    __syncwarp();
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float* pj = ps + (warp * 4 + j) * ATT_KEYS;
      for (int n = 0; n < ATT_KEYS; ++n) {
        const float p = pj[n];
#pragma unroll
        for (int k = 0; k < 4; ++k) o[j][k] = fmaf(p, xs[n * D + lane + 32 * k], o[j][k]);
      }
    }
    __syncwarp();
  }
  float ss = 0.f;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int r = r0 + 4 * warp + j;
    if (r >= N) continue;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float y = o[j][k] / l[j];
      if (Y) Y[((size_t)h * N + r) * D + lane + 32 * k] = y;
      ss = fmaf(y, y, ss);
    }
  }
  if (sq) {
#pragma unroll
    for (int off = 16; off; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    if (lane == 0) atomicAdd(sq, (double)ss);
  }
}

// E[m][n][c] = x'[n][c] - x̂'[n][c], x̂' the demotion quantiser's dequantised
// value of row n at clip ratio clips[m]: level(code)·s + z with the head's
// codebook record cb (level = code for the uniform codebook).
__global__ void __launch_bounds__(128) quant_err_kernel(const float* __restrict__ Xr, int N, int g,
                                                        const float* __restrict__ clips,
                                                        const float* __restrict__ cb, float* E) {
  __shared__ float red[8];
  const int n = blockIdx.x, m = blockIdx.y, j = threadIdx.x;
  const float x = Xr[(size_t)n * D + j];
  float mn, mx;
  group_minmax(x, j, g, red, 1, mn, mx);
  const QParams p = quant_params(mn, mx, clips[m]);
  const uint32_t code = quant_code(x, p, quant_thr(cb));
  const float lvl = fmaf(2.f * __ldg(cb + CB_BETA_HALF), (float)(code >> 1),
                         fmaf(__ldg(cb + CB_ALPHA), (float)(code & 1u), __ldg(cb + CB_C0)));
  const float xh = fmaf(lvl, __half2float(p.s), __half2float(p.z));
  E[((size_t)m * N + n) * D + j] = x - xh;
}

// err[m] += e C eᵀ for row n of E[m] (C fp32 [128][128], symmetric).
__global__ void __launch_bounds__(128) key_err_kernel(const float* __restrict__ E, int N,
                                                      const float* __restrict__ C, double* err) {
  __shared__ float es[D];
  __shared__ float part[4];
  const int n = blockIdx.x, m = blockIdx.y, c = threadIdx.x;
  es[c] = E[((size_t)m * N + n) * D + c];
  __syncthreads();
  float t = 0.f;
#pragma unroll 8
  for (int k = 0; k < D; ++k) t = fmaf(__ldg(C + k * D + c), es[k], t);
  float v = t * es[c];
#pragma unroll
  for (int off = 16; off; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  if ((c & 31) == 0) part[c >> 5] = v;
  __syncthreads();
  if (c == 0) atomicAdd(&err[m], (double)((part[0] + part[1]) + (part[2] + part[3])));
}

// Lloyd-Max codebook fit ----------------------------------------------------
// In place over rotated rows X' [N][128]: f = |t - 1.5| with t = (x - z)/s the
// quantiser's normalised value at clip ratio `clip`, or -1 where the group's
// scale is zero (no t).
__global__ void __launch_bounds__(128) fold_kernel(float* X, int g, float clip) {
  __shared__ float red[8];
  const int n = blockIdx.x, j = threadIdx.x;
  float* px = X + (size_t)n * D + j;
  const float x = *px;
  float mn, mx;
  group_minmax(x, j, g, red, 1, mn, mx);
  const QParams p = quant_params(mn, mx, clip);
  const float sf = __half2float(p.s);
  float f = -1.f;
  if (sf != 0.f) f = fabsf(__fsub_rn(__fdiv_rn(__fsub_rn(x, __half2float(p.z)), sf), 1.5f));
  *px = f;
}

// Two-level Lloyd-Max on the n folded values (one CTA): inner level a = mean
// of f <= m, outer level b = mean of f > m, m = (a + b)/2, from a = 1/2,
// b = 3/2 until the inner count repeats.  fp64 sums in a fixed order.
// out: a, b, number of centroid updates.
__global__ void __launch_bounds__(1024) lloyd_kernel(const float* __restrict__ F, int n, int max_iters,
                                                     double* out) {
  __shared__ double rs[2][32];
  __shared__ int rc[2][32];
  __shared__ double ab[2];
  __shared__ int stop;
  const int t = threadIdx.x, lane = t & 31, w = t >> 5;
  double a = 0.5, b = 1.5;
  int prev = -1, updates = 0;  // thread 0's
  for (int it = 0; it < max_iters; ++it) {
    const double m = (a + b) * 0.5;
    double si = 0.0, so = 0.0;
    int ci = 0, co = 0;
    for (int i = t; i < n; i += 1024) {
      const float f = F[i];
      if (f < 0.f) continue;
      if ((double)f <= m) {
        si += (double)f;
        ++ci;
      } else {
        so += (double)f;
        ++co;
      }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      si += __shfl_xor_sync(0xffffffffu, si, o);
      so += __shfl_xor_sync(0xffffffffu, so, o);
      ci += __shfl_xor_sync(0xffffffffu, ci, o);
      co += __shfl_xor_sync(0xffffffffu, co, o);
    }
    if (lane == 0) {
      rs[0][w] = si;
      rs[1][w] = so;
      rc[0][w] = ci;
      rc[1][w] = co;
    }
    __syncthreads();
    if (t == 0) {
      double SI = 0.0, SO = 0.0;
      int CI = 0, CO = 0;
      for (int k = 0; k < 32; ++k) {
        SI += rs[0][k];
        SO += rs[1][k];
        CI += rc[0][k];
        CO += rc[1][k];
      }
      int st = 0;
      if (CI == prev) {
        st = 1;  // same cells as last time: a and b are their centroids
      } else {
        if (CI > 0) a = SI / CI;
        if (CO > 0) b = SO / CO;
        prev = CI;
        ++updates;
      }
      ab[0] = a;
      ab[1] = b;
      stop = st;
    }
    __syncthreads();
    a = ab[0];
    b = ab[1];
    const int st = stop;
    __syncthreads();  // everyone has read ab and stop before the next round writes them
    if (st) break;
  }
  if (t == 0) {
    out[0] = a;
    out[1] = b;
    out[2] = (double)updates;
  }
}

__global__ void to_f32_kernel(const double* __restrict__ a, float* b, int n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) b[i] = (float)a[i];
}

// ----------------------------------------------------------------- cuSOLVER
struct Solver {
  bool tried = false, ok = false;
  cusolverStatus_t (*create)(cusolverDnHandle_t*) = nullptr;
  cusolverStatus_t (*destroy)(cusolverDnHandle_t) = nullptr;
  cusolverStatus_t (*set_stream)(cusolverDnHandle_t, cudaStream_t) = nullptr;
  cusolverStatus_t (*bufsize)(cusolverDnHandle_t, cusolverEigMode_t, cublasFillMode_t, int, const double*, int,
                              const double*, int*) = nullptr;
  cusolverStatus_t (*syevd)(cusolverDnHandle_t, cusolverEigMode_t, cublasFillMode_t, int, double*, int, double*,
                            double*, int, int*) = nullptr;
};

Solver& solver() {
  static Solver s;
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  if (s.tried) return s;
  s.tried = true;
  // the loader's search path first, then the toolkit's own directory (the
  // library's run path brings its cuBLAS and nvJitLink from there)
  void* h = nullptr;
  for (const char* name : {"libcusolver.so.12", "libcusolver.so", "/usr/local/cuda/lib64/libcusolver.so.12",
                           "/usr/local/cuda/lib64/libcusolver.so"}) {
    h = dlopen(name, RTLD_NOW | RTLD_LOCAL);
    if (h) break;
  }
  if (!h) return s;
  s.create = (decltype(s.create))dlsym(h, "cusolverDnCreate");
  s.destroy = (decltype(s.destroy))dlsym(h, "cusolverDnDestroy");
  s.set_stream = (decltype(s.set_stream))dlsym(h, "cusolverDnSetStream");
  s.bufsize = (decltype(s.bufsize))dlsym(h, "cusolverDnDsyevd_bufferSize");
  s.syevd = (decltype(s.syevd))dlsym(h, "cusolverDnDsyevd");
  s.ok = s.create && s.destroy && s.set_stream && s.bufsize && s.syevd;
  return s;
}

}  // namespace

CalibScratch calib_scratch_layout(int G, int N, int M) {
  CalibScratch L;
  size_t off = 0;
  auto take = [&](size_t n) {
    const size_t o = off;
    off += (n + 255) & ~(size_t)255;
    return o;
  };
  const size_t rows = (size_t)G * N;
  L.off_c = take(2 * D * D * sizeof(double));
  L.off_cf = take(D * D * sizeof(float));
  L.off_err = take(2 * (size_t)(M > 0 ? M : 1) * sizeof(double));
  L.off_clips = take((size_t)(M > 0 ? M : 1) * sizeof(float));
  L.off_y = take(rows * D * sizeof(float));   // attention output, then Q' for the clip search
  L.off_kr = take((size_t)N * D * sizeof(float));
  L.off_vr = take((size_t)N * D * sizeof(float));
  L.off_e = take((size_t)(M > 0 ? M : 1) * N * D * sizeof(float));
  L.total = off;
  return L;
}

cudaError_t calib_covariances(const __nv_bfloat16* Q, const __nv_bfloat16* K, const __nv_bfloat16* V, int G, int N,
                              uint8_t* scratch, cudaStream_t st) {
  const CalibScratch L = calib_scratch_layout(G, N, 0);
  double* C = (double*)(scratch + L.off_c);  // [0] C_Q sum, [1] C_S sum
  float* Y = (float*)(scratch + L.off_y);
  cudaError_t e = cudaMemsetAsync(C, 0, 2 * D * D * sizeof(double), st);
  if (e != cudaSuccess) return e;
  const int rows = G * N;
  gram_kernel<__nv_bfloat16><<<(rows + GRAM_ROWS - 1) / GRAM_ROWS, 256, 0, st>>>(Q, rows, C);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  e = cudaFuncSetAttribute(causal_attn_kernel<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize, ATT_SMEM);
  if (e != cudaSuccess) return e;
  causal_attn_kernel<__nv_bfloat16><<<dim3((N + ATT_ROWS - 1) / ATT_ROWS, G), 256, ATT_SMEM, st>>>(Q, K, V, N, Y,
                                                                                                   nullptr);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  gram_kernel<float><<<(rows + GRAM_ROWS - 1) / GRAM_ROWS, 256, 0, st>>>(Y, rows, C + D * D);
  return cudaGetLastError();
}

// The cuSOLVER handle and the device buffers of the 128x128 problem are made
// once and reused while the calls stay on the same device; a call on another
// device makes them again there (the old ones are released).
struct EighState {
  int device = -1;
  cusolverDnHandle_t hd = nullptr;
  double *A = nullptr, *W = nullptr, *work = nullptr;
  int* info = nullptr;
  int lwork = 0;
};

oscar_status calib_eigh(const double* dC, double* evec_host, cudaStream_t st, int* cuda_err) {
  Solver& s = solver();
  if (!s.ok) return OSCAR_ERR_UNSUPPORTED;
  static EighState es;
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  cudaError_t e = cudaSuccess;
  int dev = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) {
    *cuda_err = (int)e;
    return OSCAR_ERR_CUDA;
  }
  auto release = [&](EighState& x) {  // on the device that owns x
    if (!x.hd && !x.A && !x.W && !x.work && !x.info) return;
    int cur = 0;
    cudaGetDevice(&cur);
    if (x.device >= 0) cudaSetDevice(x.device);
    if (x.hd) s.destroy(x.hd);
    cudaFree(x.A);
    cudaFree(x.W);
    cudaFree(x.work);
    cudaFree(x.info);
    cudaSetDevice(cur);
    x = EighState();
  };
  if (es.hd && es.device != dev) release(es);
  if (!es.hd) {  // build the state whole, or leave none
    EighState n;
    n.device = dev;
    if (s.create(&n.hd) != CUSOLVER_STATUS_SUCCESS) {
      *cuda_err = 0;
      return OSCAR_ERR_CUDA;
    }
    e = cudaMalloc((void**)&n.A, D * D * sizeof(double));
    if (e == cudaSuccess) e = cudaMalloc((void**)&n.W, D * sizeof(double));
    if (e == cudaSuccess) e = cudaMalloc((void**)&n.info, sizeof(int));
    bool ok = e == cudaSuccess &&
              s.bufsize(n.hd, CUSOLVER_EIG_MODE_VECTOR, CUBLAS_FILL_MODE_LOWER, D, n.A, D, n.W, &n.lwork) ==
                  CUSOLVER_STATUS_SUCCESS;
    if (ok) e = cudaMalloc((void**)&n.work, (size_t)(n.lwork > 0 ? n.lwork : 1) * sizeof(double));
    ok = ok && e == cudaSuccess;
    if (!ok) {
      release(n);
      *cuda_err = (int)e;
      return OSCAR_ERR_CUDA;
    }
    es = n;
  }
  int hinfo = 0;
  oscar_status status = OSCAR_OK;
  e = cudaMemcpyAsync(es.A, dC, D * D * sizeof(double), cudaMemcpyDeviceToDevice, st);
  if (e == cudaSuccess && s.set_stream(es.hd, st) != CUSOLVER_STATUS_SUCCESS) status = OSCAR_ERR_CUDA;
  if (e == cudaSuccess && status == OSCAR_OK &&
      s.syevd(es.hd, CUSOLVER_EIG_MODE_VECTOR, CUBLAS_FILL_MODE_LOWER, D, es.A, D, es.W, es.work, es.lwork,
              es.info) != CUSOLVER_STATUS_SUCCESS)
    status = OSCAR_ERR_CUDA;
  if (e == cudaSuccess && status == OSCAR_OK)
    e = cudaMemcpyAsync(evec_host, es.A, D * D * sizeof(double), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess && status == OSCAR_OK) e = cudaMemcpyAsync(&hinfo, es.info, sizeof(int), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) {
    *cuda_err = (int)e;
    return OSCAR_ERR_CUDA;
  }
  if (status == OSCAR_OK && hinfo != 0) status = OSCAR_ERR_STATE;
  return status;
}

cudaError_t calib_clip_errors(const float* R_K, const float* R_V, const __nv_bfloat16* Q, const __nv_bfloat16* K,
                              const __nv_bfloat16* V, int G, int N, int g, const float* clips_host, int M,
                              const float* cb_k, const float* cb_v, uint8_t* scratch, cudaStream_t st) {
  const CalibScratch L = calib_scratch_layout(G, N, M);
  double* C = (double*)(scratch + L.off_c);
  float* Cf = (float*)(scratch + L.off_cf);
  double* err = (double*)(scratch + L.off_err);
  float* clips = (float*)(scratch + L.off_clips);
  float* Qr = (float*)(scratch + L.off_y);
  float* Kr = (float*)(scratch + L.off_kr);
  float* Vr = (float*)(scratch + L.off_vr);
  float* E = (float*)(scratch + L.off_e);
  const int rows = G * N;
  cudaError_t e = cudaMemsetAsync(C, 0, D * D * sizeof(double), st);
  if (e == cudaSuccess) e = cudaMemsetAsync(err, 0, 2 * (size_t)M * sizeof(double), st);
  if (e == cudaSuccess) e = cudaMemcpyAsync(clips, clips_host, (size_t)M * sizeof(float), cudaMemcpyHostToDevice, st);
  // rotated calibration queries, keys and values (the demotion's fp32 rotation)
  if (e == cudaSuccess) e = launch_debug_rotate(R_K, Q, Qr, rows, st);
  if (e == cudaSuccess) e = launch_debug_rotate(R_K, K, Kr, N, st);
  if (e == cudaSuccess) e = launch_debug_rotate(R_V, V, Vr, N, st);
  if (e != cudaSuccess) return e;
  // keys: Σ_n e_n (Q'ᵀQ') e_nᵀ
  gram_kernel<float><<<(rows + GRAM_ROWS - 1) / GRAM_ROWS, 256, 0, st>>>(Qr, rows, C);
  to_f32_kernel<<<(D * D + 255) / 256, 256, 0, st>>>(C, Cf, D * D);
  quant_err_kernel<<<dim3(N, M), 128, 0, st>>>(Kr, N, g, clips, cb_k, E);
  key_err_kernel<<<dim3(N, M), 128, 0, st>>>(E, N, Cf, err);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  // values: Σ_h ||S_h E_m||²_F
  quant_err_kernel<<<dim3(N, M), 128, 0, st>>>(Vr, N, g, clips, cb_v, E);
  e = cudaFuncSetAttribute(causal_attn_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, ATT_SMEM);
  if (e != cudaSuccess) return e;
  for (int m = 0; m < M; ++m) {
    causal_attn_kernel<float><<<dim3((N + ATT_ROWS - 1) / ATT_ROWS, G), 256, ATT_SMEM, st>>>(
        Q, K, E + (size_t)m * N * D, N, nullptr, err + M + m);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

size_t codebook_scratch_bytes(int N) { return ((size_t)N * D * 4 + 255) / 256 * 256 + 256; }

cudaError_t calib_fit_codebook(const float* R, const __nv_bfloat16* X, int N, int g, float clip, int max_iters,
                               uint8_t* scratch, double* ab_host, int* updates_host, cudaStream_t st) {
  float* F = (float*)scratch;
  double* out = (double*)(scratch + ((size_t)N * D * 4 + 255) / 256 * 256);
  cudaError_t e = launch_debug_rotate(R, X, F, N, st);  // the demotion's fp32 rotation
  if (e != cudaSuccess) return e;
  fold_kernel<<<N, 128, 0, st>>>(F, g, clip);
  lloyd_kernel<<<1, 1024, 0, st>>>(F, N * D, max_iters, out);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  double h[3];
  e = cudaMemcpyAsync(h, out, sizeof(h), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return e;
  ab_host[0] = h[0];
  ab_host[1] = h[1];
  *updates_host = (int)h[2];
  return cudaSuccess;
}

}  // namespace oscar
