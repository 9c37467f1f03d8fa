// Output side and sampler of one denoiser evaluation: the shifted sigma grid,
// the data-ward Euler step, the conditioning noise mix, row selection, the
// final AdaLN table of a modality and the FP32 velocity head.
//
// Sampler arithmetic follows the RFC's scheduler fingerprint (section 2) in
// IEEE fp32 with one rounding per written operation, in the written order:
// every product, sum and quotient below is an explicit _rn intrinsic, so the
// compiler cannot contract or reorder them and the results are the same bits
// on every run.  The final layer's FP32 modules (RFC section 5,
// final_adaln_out and the video/audio output projections) accumulate in fp32
// in a fixed order.
#include "h3_device.cuh"
#include "h3_internal.h"

#include <cmath>

namespace h3 {

namespace {

// value i of the grid before collapsing duplicates: the shifted linspace point
// for i < n, the terminal zero for i == n
__device__ __forceinline__ float grid_value(int i, int n, float s) {
  if (i >= n) return 0.0f;
  const double lin = __dsub_rn(1.0, __ddiv_rn((double)i, (double)(n - 1)));
  const float sg = __double2float_rn(lin);
  const float num = __fmul_rn(s, sg);
  const float den = __fadd_rn(1.0f, __fmul_rn(__fsub_rn(s, 1.0f), sg));
  return __fdiv_rn(num, den);
}

// Exclusive scan of one flag per thread over a 1024-thread block; returns the
// thread's offset and writes the block total to *total.
__device__ __forceinline__ int block_exclusive_scan(int flag, int* warp_sums, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = flag;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = lane < (int)(blockDim.x >> 5) ? warp_sums[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += v;
    }
    warp_sums[lane] = w;   // inclusive over warps
  }
  __syncthreads();
  const int before = warp > 0 ? warp_sums[warp - 1] : 0;
  *total = warp_sums[(blockDim.x >> 5) - 1];
  const int r = before + incl - flag;
  __syncthreads();
  return r;
}

}  // namespace

// One block of 1024 threads walks the n + 1 candidate values in chunks; a
// value is kept when it differs from its predecessor (each thread recomputes
// the predecessor itself, the values being a pure function of the index).
__global__ void __launch_bounds__(1024) sigma_grid_kernel(int n, float s, float* __restrict__ sigmas,
                                                          int32_t* __restrict__ count) {
  griddep_launch_dependents();
  griddep_wait();
  __shared__ int warp_sums[32];
  int base = 0;
  for (int c = 0; c <= n; c += blockDim.x) {
    const int i = c + (int)threadIdx.x;
    float v = 0.0f;
    int keep = 0;
    if (i <= n) {
      v = grid_value(i, n, s);
      keep = (i == 0) || (v != grid_value(i - 1, n, s));
    }
    int total;
    const int pos = block_exclusive_scan(keep, warp_sums, &total);
    if (keep) sigmas[base + pos] = v;
    base += total;
  }
  if (threadIdx.x == 0) *count = base;
}

// x_next = r*xt + (1-r)*(xt + sigma*v), r = sigma_next / sigma
// out may alias xt (an in-place step): no restrict qualifiers on them
__global__ void __launch_bounds__(256) ode_step_kernel(long long n, const float* xt, const float* v, float sigma,
                                                       float sigma_next, float* out) {
  griddep_launch_dependents();
  griddep_wait();
  const float r = __fdiv_rn(sigma_next, sigma);
  const float omr = __fsub_rn(1.0f, r);
  auto one = [&](float x, float vv) {
    const float x0 = __fadd_rn(x, __fmul_rn(sigma, vv));
    return __fadd_rn(__fmul_rn(r, x), __fmul_rn(omr, x0));
  };
  const long long n4 = n >> 2;
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long q = (long long)blockIdx.x * blockDim.x + threadIdx.x; q < n4; q += stride) {
    const float4 a = reinterpret_cast<const float4*>(xt)[q];
    const float4 b = reinterpret_cast<const float4*>(v)[q];
    reinterpret_cast<float4*>(out)[q] = make_float4(one(a.x, b.x), one(a.y, b.y), one(a.z, b.z), one(a.w, b.w));
  }
  for (long long i = (n4 << 2) + (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride)
    out[i] = one(xt[i], v[i]);
}

// t*x0 + (1-t)*noise
__global__ void __launch_bounds__(256) noise_mix_kernel(long long n, const float* x0, const float* noise, float t,
                                                        float* out) {
  griddep_launch_dependents();
  griddep_wait();
  const float omt = __fsub_rn(1.0f, t);
  auto one = [&](float a, float b) { return __fadd_rn(__fmul_rn(t, a), __fmul_rn(omt, b)); };
  const long long n4 = n >> 2;
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long q = (long long)blockIdx.x * blockDim.x + threadIdx.x; q < n4; q += stride) {
    const float4 a = reinterpret_cast<const float4*>(x0)[q];
    const float4 b = reinterpret_cast<const float4*>(noise)[q];
    reinterpret_cast<float4*>(out)[q] = make_float4(one(a.x, b.x), one(a.y, b.y), one(a.z, b.z), one(a.w, b.w));
  }
  for (long long i = (n4 << 2) + (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride)
    out[i] = one(x0[i], noise[i]);
}

// Stable compaction of the rows whose tag equals `tag` (one block).
__global__ void __launch_bounds__(1024) select_rows_kernel(int n, const int32_t* __restrict__ tags, int tag,
                                                           int32_t* __restrict__ rows, int32_t* __restrict__ count) {
  griddep_launch_dependents();
  griddep_wait();
  __shared__ int warp_sums[32];
  int base = 0;
  for (int c = 0; c < n; c += blockDim.x) {
    const int i = c + (int)threadIdx.x;
    const int keep = (i < n && tags[i] == tag) ? 1 : 0;
    int total;
    const int pos = block_exclusive_scan(keep, warp_sums, &total);
    if (keep) rows[base + pos] = i;
    base += total;
  }
  if (threadIdx.x == 0) *count = base;
}

// ---------------------------------------------------------------------------
// final AdaLN table: out[t][j] = SiLU(t_cond[t]) . w[j] + b[j], fp32, j < 2D.
// Each CTA holds u = SiLU(t_cond) [T][C] in shared memory; each warp owns one
// weight row at a time and streams it with 16-byte loads, four in flight per
// lane (lane l takes float4 columns l + 32i), keeping T running sums that it
// reduces over the warp with a fixed xor tree.  Many CTAs per SM keep enough
// bytes in flight for HBM; the kernel is bound by the 2D x C fp32 weights.
// ---------------------------------------------------------------------------
constexpr int FA_THREADS = 256;

__global__ void __launch_bounds__(FA_THREADS) final_adaln_kernel(const float* __restrict__ w,
                                                                 const float* __restrict__ b,
                                                                 const float* __restrict__ t_cond, int T, int C,
                                                                 int rows, float* __restrict__ out) {
  extern __shared__ float u[];   // [T][C]
  griddep_launch_dependents();
  griddep_wait();
  for (int i = threadIdx.x; i < T * C; i += blockDim.x) {
    const float x = t_cond[i];
    u[i] = x / (1.0f + expf(-x));
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nw = blockDim.x >> 5;
  const int c4 = C >> 2;
  for (int j = blockIdx.x * nw + warp; j < rows; j += gridDim.x * nw) {
    const float4* wr = reinterpret_cast<const float4*>(w + (size_t)j * C);
    float acc[16];
#pragma unroll
    for (int t = 0; t < 16; ++t) acc[t] = 0.0f;
    for (int k4 = lane; k4 < c4; k4 += 4 * 32) {
      float4 wv[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int kk = k4 + q * 32;
        wv[q] = kk < c4 ? __ldg(wr + kk) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int kk = k4 + q * 32;
        if (kk < c4) {
#pragma unroll
          for (int t = 0; t < 16; ++t) {
            if (t < T) {
              const float4 uv = reinterpret_cast<const float4*>(u + t * C)[kk];
              acc[t] = __fmaf_rn(uv.x, wv[q].x, acc[t]);
              acc[t] = __fmaf_rn(uv.y, wv[q].y, acc[t]);
              acc[t] = __fmaf_rn(uv.z, wv[q].z, acc[t]);
              acc[t] = __fmaf_rn(uv.w, wv[q].w, acc[t]);
            }
          }
        }
      }
    }
#pragma unroll
    for (int t = 0; t < 16; ++t) {
      if (t < T) {
        float a = acc[t];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
        if (lane == 0) out[(size_t)t * rows + j] = a + (b ? b[j] : 0.0f);
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Velocity head.  A CTA takes 64 selected rows and all P columns (P padded to
// 16 * PT, PT in {2, 4, 6, 8}).  Phase 1: the inverse RMS of each row (fp32,
// lane partial sums then a fixed xor tree).  Phase 2 walks D in 32-column
// chunks: the modulated activations a[k][row] = (x * inv) * (1 + scale) +
// shift and the head chunk w[k][p] are staged in shared memory (16-byte global
// loads; the next chunk's loads are issued before the current chunk is
// multiplied), and thread (ty, tx) keeps a 4-row x PT-column register tile,
// reading 4 rows with one 16-byte and its PT columns with 8-byte shared loads
// per k, and accumulating in k order.  Rows whose metadata is out of range are
// reported and left unwritten.
// ---------------------------------------------------------------------------
constexpr int OH_ROWS = 64, OH_KC = 32, OH_THREADS = 256;

template <int PT>
__global__ void __launch_bounds__(OH_THREADS) output_head_kernel(const OutputHeadArgs a) {
  constexpr int PW = 16 * PT;        // padded head width
  constexpr int WS = PW + 2;         // s_w row stride (even, 2 mod 32)
  __shared__ __align__(16) float s_a[OH_KC][OH_ROWS];
  __shared__ __align__(16) float s_w[OH_KC * WS];
  __shared__ float s_inv[OH_ROWS];
  __shared__ int s_row[OH_ROWS], s_t[OH_ROWS];
  griddep_launch_dependents();
  griddep_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int i0 = blockIdx.x * OH_ROWS;
  const int D = a.D, P = a.P;
  if (threadIdx.x < OH_ROWS) {
    const int i = i0 + (int)threadIdx.x;
    int r = -1, t = 0;
    if (i < a.n_sel) {
      r = a.rows[i];
      if ((unsigned)r >= (unsigned)a.S) {
        record_error(a.err, DEVERR_INDEX);
        r = -1;
      } else {
        t = a.tidx[r];
        if ((unsigned)t >= (unsigned)a.T) {
          record_error(a.err, DEVERR_INDEX);
          r = -1;
          t = 0;
        }
      }
    }
    s_row[threadIdx.x] = r;
    s_t[threadIdx.x] = t;
  }
  __syncthreads();
  // phase 1: inverse RMS, eight rows per warp
  for (int rr = warp; rr < OH_ROWS; rr += OH_THREADS / 32) {
    const int r = s_row[rr];
    float ss = 0.0f;
    if (r >= 0) {
      const uint4* xr = reinterpret_cast<const uint4*>(a.x + (size_t)r * D);
      for (int c = lane; c < (D >> 3); c += 32) {
        const uint4 q = xr[c];
        const uint32_t wv[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float lo = bf16_lo(wv[e]), hi = bf16_hi(wv[e]);
          ss = __fmaf_rn(lo, lo, ss);
          ss = __fmaf_rn(hi, hi, ss);
        }
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if (lane == 0) s_inv[rr] = 1.0f / sqrtf(ss / (float)D + a.eps);
  }
  __syncthreads();

  // staging roles.  activations: row ar = tid / 4, columns ak..ak+7 of the chunk;
  // head: float4 slots f = tid + 256 e over PW rows x 8 float4 (rows >= P are zero)
  const int ar = threadIdx.x >> 2, ak = (threadIdx.x & 3) * 8;
  const int my_row = s_row[ar];
  const float my_inv = s_inv[ar];
  const float* tab = a.table + (size_t)s_t[ar] * 2 * D;
  constexpr int WSLOTS = (PW * (OH_KC / 4) + OH_THREADS - 1) / OH_THREADS;
  auto load_chunk = [&](int k0, uint4& xv, float4 (&sh)[2], float4 (&sc)[2], float4 (&wv)[WSLOTS]) {
    if (my_row >= 0) {
      xv = *reinterpret_cast<const uint4*>(a.x + (size_t)my_row * D + k0 + ak);
      sh[0] = *reinterpret_cast<const float4*>(tab + k0 + ak);
      sh[1] = *reinterpret_cast<const float4*>(tab + k0 + ak + 4);
      sc[0] = *reinterpret_cast<const float4*>(tab + D + k0 + ak);
      sc[1] = *reinterpret_cast<const float4*>(tab + D + k0 + ak + 4);
    }
#pragma unroll
    for (int e = 0; e < WSLOTS; ++e) {
      const int f = (int)threadIdx.x + e * OH_THREADS;
      const int p = f / (OH_KC / 4), kq = f % (OH_KC / 4);
      wv[e] = (p < P) ? *reinterpret_cast<const float4*>(a.w + (size_t)p * D + k0 + kq * 4)
                      : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  };
  auto store_chunk = [&](const uint4& xv, const float4 (&sh)[2], const float4 (&sc)[2],
                         const float4 (&wv)[WSLOTS]) {
    const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
    const float shv[8] = {sh[0].x, sh[0].y, sh[0].z, sh[0].w, sh[1].x, sh[1].y, sh[1].z, sh[1].w};
    const float scv[8] = {sc[0].x, sc[0].y, sc[0].z, sc[0].w, sc[1].x, sc[1].y, sc[1].z, sc[1].w};
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      float val = 0.0f;
      if (my_row >= 0) {
        const float xvv = (e & 1) ? bf16_hi(xw[e >> 1]) : bf16_lo(xw[e >> 1]);
        val = __fmaf_rn(xvv * my_inv, 1.0f + scv[e], shv[e]);
      }
      s_a[ak + e][ar] = val;
    }
#pragma unroll
    for (int e = 0; e < WSLOTS; ++e) {
      const int f = (int)threadIdx.x + e * OH_THREADS;
      const int p = f / (OH_KC / 4), kq = f % (OH_KC / 4);
      if (p < PW) {
        s_w[(kq * 4 + 0) * WS + p] = wv[e].x;
        s_w[(kq * 4 + 1) * WS + p] = wv[e].y;
        s_w[(kq * 4 + 2) * WS + p] = wv[e].z;
        s_w[(kq * 4 + 3) * WS + p] = wv[e].w;
      }
    }
  };

  const int ty = threadIdx.x >> 4, tx = threadIdx.x & 15;   // rows 4ty..4ty+3, columns PT tx..PT tx+PT-1
  float acc[4][PT];
#pragma unroll
  for (int r4 = 0; r4 < 4; ++r4)
#pragma unroll
    for (int c = 0; c < PT; ++c) acc[r4][c] = 0.0f;
  uint4 xv = make_uint4(0u, 0u, 0u, 0u);
  float4 sh[2], sc[2], wv[WSLOTS];
  load_chunk(0, xv, sh, sc, wv);
  for (int k0 = 0; k0 < D; k0 += OH_KC) {
    store_chunk(xv, sh, sc, wv);
    __syncthreads();
    if (k0 + OH_KC < D) load_chunk(k0 + OH_KC, xv, sh, sc, wv);   // in flight during the products
#pragma unroll 8
    for (int kk = 0; kk < OH_KC; ++kk) {
      const float4 av = *reinterpret_cast<const float4*>(&s_a[kk][ty * 4]);
      float w[PT];
#pragma unroll
      for (int m = 0; m < PT / 2; ++m) {
        const float2 w2 = *reinterpret_cast<const float2*>(&s_w[kk * WS + tx * PT + 2 * m]);
        w[2 * m] = w2.x;
        w[2 * m + 1] = w2.y;
      }
      const float a4[4] = {av.x, av.y, av.z, av.w};
#pragma unroll
      for (int r4 = 0; r4 < 4; ++r4)
#pragma unroll
        for (int c = 0; c < PT; ++c) acc[r4][c] = __fmaf_rn(a4[r4], w[c], acc[r4][c]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int r4 = 0; r4 < 4; ++r4) {
    const int rr = ty * 4 + r4;
    const int i = i0 + rr;
    if (s_row[rr] >= 0 && i < a.n_sel) {
#pragma unroll
      for (int c = 0; c < PT; ++c) {
        const int p = tx * PT + c;
        if (p < P) a.out[(size_t)i * P + p] = acc[r4][c] + (a.b ? a.b[p] : 0.0f);
      }
    }
  }
}

// ---------------------------------------------------------------------------
// launchers
// ---------------------------------------------------------------------------
cudaError_t launch_sigma_grid(int n, float s, float* sigmas, int32_t* count, cudaStream_t st) {
  cudaError_t e = launch_kernel(sigma_grid_kernel, dim3(1), dim3(1024), 0, st, n, s, sigmas, count);
  if (e != cudaSuccess) return e;
  set_kernel_info("sigma_grid_kernel fp32 one-rounding-per-op points=%d shift=%g", n, (double)s);
  return cudaGetLastError();
}

static int elementwise_grid(long long n) {
  const long long blocks = (n / 4 + 255) / 256;
  const long long cap = 8LL * num_sms();
  return (int)(blocks < 1 ? 1 : (blocks > cap ? cap : blocks));
}

cudaError_t launch_ode_step(long long n, const float* xt, const float* v, float sigma, float sigma_next, float* out,
                            cudaStream_t st) {
  cudaError_t e = launch_kernel(ode_step_kernel, dim3(elementwise_grid(n)), dim3(256), 0, st, n, xt, v, sigma,
                                sigma_next, out);
  if (e != cudaSuccess) return e;
  set_kernel_info("ode_step_kernel fp32 float4 n=%lld", n);
  return cudaGetLastError();
}

cudaError_t launch_noise_mix(long long n, const float* x0, const float* noise, float t, float* out, cudaStream_t st) {
  cudaError_t e = launch_kernel(noise_mix_kernel, dim3(elementwise_grid(n)), dim3(256), 0, st, n, x0, noise, t, out);
  if (e != cudaSuccess) return e;
  set_kernel_info("noise_mix_kernel fp32 float4 n=%lld", n);
  return cudaGetLastError();
}

cudaError_t launch_select_rows(int n, const int32_t* tags, int tag, int32_t* rows, int32_t* count, cudaStream_t st) {
  cudaError_t e = launch_kernel(select_rows_kernel, dim3(1), dim3(1024), 0, st, n, tags, tag, rows, count);
  if (e != cudaSuccess) return e;
  set_kernel_info("select_rows_kernel stable-compaction rows=%d tag=%d", n, tag);
  return cudaGetLastError();
}

cudaError_t launch_final_adaln(const float* w, const float* b, const float* t_cond, int T, int C, int rows,
                               float* out, cudaStream_t st) {
  const int smem = T * C * (int)sizeof(float);
  cudaError_t e = cudaFuncSetAttribute(final_adaln_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int warps = FA_THREADS / 32;
  int grid = (rows + warps - 1) / warps;
  if (grid > 8 * num_sms()) grid = 8 * num_sms();
  e = launch_kernel(final_adaln_kernel, dim3(grid), dim3(FA_THREADS), (size_t)smem, st, w, b, t_cond, T, C, rows,
                    out);
  if (e != cudaSuccess) return e;
  set_kernel_info("final_adaln_kernel fp32 warp-per-row T=%d C=%d rows=%d grid=%d", T, C, rows, grid);
  return cudaGetLastError();
}

cudaError_t launch_output_head(const OutputHeadArgs& a, cudaStream_t st) {
  const int grid = (a.n_sel + OH_ROWS - 1) / OH_ROWS;
  const int pt = a.P <= 32 ? 2 : (a.P <= 64 ? 4 : (a.P <= 96 ? 6 : 8));
  cudaError_t e;
  switch (pt) {
    case 2: e = launch_kernel(output_head_kernel<2>, dim3(grid), dim3(OH_THREADS), 0, st, a); break;
    case 4: e = launch_kernel(output_head_kernel<4>, dim3(grid), dim3(OH_THREADS), 0, st, a); break;
    case 6: e = launch_kernel(output_head_kernel<6>, dim3(grid), dim3(OH_THREADS), 0, st, a); break;
    default: e = launch_kernel(output_head_kernel<8>, dim3(grid), dim3(OH_THREADS), 0, st, a); break;
  }
  if (e != cudaSuccess) return e;
  set_kernel_info("output_head_kernel<%d> fp32 rows/cta=%d k_chunk=%d reg-tile=4x%d P=%d rows=%d", pt, OH_ROWS,
                  OH_KC, pt, a.P, a.n_sel);
  return cudaGetLastError();
}

}  // namespace h3
