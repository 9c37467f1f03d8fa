// Input side of one denoiser evaluation: the (1, 2, 2) patch permutation of
// the video latent and its inverse, the FP32 video/audio input projections
// rounded once to bf16 and written into the packed residual stream at their
// destination rows, the row scatter of already-projected bf16 rows, and the
// FP32 timestep sinusoid and MLP that produce the conditioning rows (RFC
// section 2 input/conditioning and mixed-precision fingerprints; section 5
// video_patch_pack_unpack, video/audio_input_projection_fp32,
// packed_index_copy, timestep_sinusoid_h3, timestep_mlp_fp32).
#include "h3_device.cuh"
#include "h3_internal.h"

#include <cmath>

namespace h3 {

// rows [T*(H/2)*(W/2)][C*4], row (t, hh, ww) t slowest, feature (c, a, b) c
// slowest.  pack: dst (rows) [i] = src (latent) [li]; unpack: dst (latent)
// [li] = src (rows) [i], with i the row-major position in the rows.
__global__ void __launch_bounds__(256) patch_pack_kernel(int C, int T, int H, int W, const float* __restrict__ src,
                                                         float* __restrict__ dst, int unpack) {
  griddep_launch_dependents();
  griddep_wait();
  const int H2 = H >> 1, W2 = W >> 1, F = C * 4;
  const long long n = (long long)T * H2 * W2 * F;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x) {
    const int f = (int)(i % F);
    const long long r = i / F;
    const int ww = (int)(r % W2), hh = (int)((r / W2) % H2), t = (int)(r / ((long long)W2 * H2));
    const int c = f >> 2, a = (f >> 1) & 1, b = f & 1;
    const long long li = (((long long)c * T + t) * H + (2 * hh + a)) * W + (2 * ww + b);
    if (unpack)
      dst[li] = src[i];
    else
      dst[i] = src[li];
  }
}

// ---------------------------------------------------------------------------
// FP32 input projection: out[dst[i]][j] = bf16(src[i] . w[j] + b[j]).  A CTA
// takes 128 source rows x 128 output columns with the whole K (<= 128) staged
// in shared memory, transposed so that a thread reads its 8 rows and its 8
// columns with two 16-byte loads each per k; 8x8 register tile per thread,
// accumulated in k order.
// ---------------------------------------------------------------------------
constexpr int IP_ROWS = 128, IP_COLS = 128, IP_THREADS = 256;

__global__ void __launch_bounds__(IP_THREADS) input_proj_kernel(const InputProjArgs a) {
  extern __shared__ __align__(16) float ip_smem[];
  float* s_x = ip_smem;                       // [K][128 rows]
  float* s_w = ip_smem + a.K * IP_ROWS;       // [K][128 cols]
  griddep_launch_dependents();
  griddep_wait();
  const int r0 = blockIdx.x * IP_ROWS, c0 = blockIdx.y * IP_COLS;
  const int k4n = a.K >> 2;
  // consecutive threads take consecutive rows of one k-quad, so the transposed
  // shared stores of a warp fall in 32 different banks
  for (int idx = threadIdx.x; idx < IP_ROWS * k4n; idx += IP_THREADS) {
    const int r = idx % IP_ROWS, k4 = idx / IP_ROWS;
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (r0 + r < a.n) v = *reinterpret_cast<const float4*>(a.src + (size_t)(r0 + r) * a.K + 4 * k4);
    s_x[(4 * k4 + 0) * IP_ROWS + r] = v.x;
    s_x[(4 * k4 + 1) * IP_ROWS + r] = v.y;
    s_x[(4 * k4 + 2) * IP_ROWS + r] = v.z;
    s_x[(4 * k4 + 3) * IP_ROWS + r] = v.w;
  }
  for (int idx = threadIdx.x; idx < IP_COLS * k4n; idx += IP_THREADS) {
    const int c = idx % IP_COLS, k4 = idx / IP_COLS;
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (c0 + c < a.D) v = *reinterpret_cast<const float4*>(a.w + (size_t)(c0 + c) * a.K + 4 * k4);
    s_w[(4 * k4 + 0) * IP_COLS + c] = v.x;
    s_w[(4 * k4 + 1) * IP_COLS + c] = v.y;
    s_w[(4 * k4 + 2) * IP_COLS + c] = v.z;
    s_w[(4 * k4 + 3) * IP_COLS + c] = v.w;
  }
  __syncthreads();
  const int ty = threadIdx.x >> 4, tx = threadIdx.x & 15;
  float acc[8][8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = 0.0f;
#pragma unroll 2
  for (int k = 0; k < a.K; ++k) {
    const float4 x0 = *reinterpret_cast<const float4*>(s_x + k * IP_ROWS + ty * 8);
    const float4 x1 = *reinterpret_cast<const float4*>(s_x + k * IP_ROWS + ty * 8 + 4);
    const float4 w0 = *reinterpret_cast<const float4*>(s_w + k * IP_COLS + tx * 8);
    const float4 w1 = *reinterpret_cast<const float4*>(s_w + k * IP_COLS + tx * 8 + 4);
    const float xr[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
    const float wc[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[i][j] = __fmaf_rn(xr[i], wc[j], acc[i][j]);
  }
  const int c = c0 + tx * 8;
  if (c >= a.D) return;
  float bias[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) bias[j] = a.b ? a.b[c + j] : 0.0f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int r = r0 + ty * 8 + i;
    if (r >= a.n) continue;
    const int d = a.dst[r];
    if ((unsigned)d >= (unsigned)a.n_dst) {
      record_error(a.err, DEVERR_INDEX);
      continue;
    }
    uint4 o;
    o.x = pack_bf16x2(acc[i][0] + bias[0], acc[i][1] + bias[1]);
    o.y = pack_bf16x2(acc[i][2] + bias[2], acc[i][3] + bias[3]);
    o.z = pack_bf16x2(acc[i][4] + bias[4], acc[i][5] + bias[5]);
    o.w = pack_bf16x2(acc[i][6] + bias[6], acc[i][7] + bias[7]);
    *reinterpret_cast<uint4*>(a.out + (size_t)d * a.D + c) = o;
  }
}

// out[dst[i]] = src[i] for bf16 rows of D (16-byte copies); one warp per row
__global__ void __launch_bounds__(256) index_copy_kernel(int n, int D, const __nv_bfloat16* __restrict__ src,
                                                         const int32_t* __restrict__ dst, int n_dst,
                                                         __nv_bfloat16* __restrict__ out, uint32_t* err) {
  griddep_launch_dependents();
  griddep_wait();
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  const int nw = (gridDim.x * blockDim.x) >> 5;
  for (int r = warp; r < n; r += nw) {
    const int d = dst[r];
    if ((unsigned)d >= (unsigned)n_dst) {
      if (lane == 0) record_error(err, DEVERR_INDEX);
      continue;
    }
    const uint4* s = reinterpret_cast<const uint4*>(src + (size_t)r * D);
    uint4* o = reinterpret_cast<uint4*>(out + (size_t)d * D);
    for (int c = lane; c < (D >> 3); c += 32) o[c] = s[c];
  }
}

// ---------------------------------------------------------------------------
// timestep features: e[t][i] = cos(t f_i), e[t][128 + i] = sin(t f_i),
// f_i = exp(-ln(10000) i / 128), fp32
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) sinusoid_kernel(int T, const float* __restrict__ t, float* __restrict__ e) {
  griddep_launch_dependents();
  griddep_wait();
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= T * 128) return;
  const int row = i >> 7, k = i & 127;
  const float f = expf(-logf(10000.0f) * ((float)k / 128.0f));
  const float ang = t[row] * f;
  float s, c;
  sincosf(ang, &s, &c);
  e[row * 256 + k] = c;
  e[row * 256 + 128 + k] = s;
}

// ---------------------------------------------------------------------------
// Skinny FP32 linear for a few rows: out[t][j] = act(in[t] . w[j] + b[j]),
// t < T <= 16.  One warp per output column j streams w[j] with 16-byte loads
// (four in flight per lane) against the inputs read through the read-only
// cache, keeps T running sums and reduces them with a fixed xor tree.
// act: 0 none, 1 SiLU.  Bound by the fp32 weight stream.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) rows_linear_kernel(int T, int K, int N, const float* __restrict__ in,
                                                          const float* __restrict__ w, const float* __restrict__ b,
                                                          int act, float* __restrict__ out) {
  griddep_launch_dependents();
  griddep_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nw = blockDim.x >> 5;
  const int k4n = K >> 2;
  for (int j = blockIdx.x * nw + warp; j < N; j += gridDim.x * nw) {
    const float4* wr = reinterpret_cast<const float4*>(w + (size_t)j * K);
    float acc[16];
#pragma unroll
    for (int t = 0; t < 16; ++t) acc[t] = 0.0f;
    for (int k4 = lane; k4 < k4n; k4 += 4 * 32) {
      float4 wv[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int kk = k4 + q * 32;
        wv[q] = kk < k4n ? __ldg(wr + kk) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int kk = k4 + q * 32;
        if (kk < k4n) {
#pragma unroll
          for (int t = 0; t < 16; ++t) {
            if (t < T) {
              const float4 uv = __ldg(reinterpret_cast<const float4*>(in + (size_t)t * K) + kk);
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
        float v = acc[t];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == 0) {
          v += b ? b[j] : 0.0f;
          if (act == 1) v = v / (1.0f + expf(-v));
          out[(size_t)t * N + j] = v;
        }
      }
    }
  }
}

// ---------------------------------------------------------------------------
// launchers
// ---------------------------------------------------------------------------
static int grid_for(long long work, int per_block, int cap_per_sm) {
  long long g = (work + per_block - 1) / per_block;
  const long long cap = (long long)cap_per_sm * num_sms();
  return (int)(g < 1 ? 1 : (g > cap ? cap : g));
}

cudaError_t launch_patch_pack(int C, int T, int H, int W, const float* src, float* dst, bool unpack,
                              cudaStream_t st) {
  const long long n = (long long)C * T * H * W;
  cudaError_t e = launch_kernel(patch_pack_kernel, dim3(grid_for(n, 256, 16)), dim3(256), 0, st, C, T, H, W, src,
                                dst, unpack ? 1 : 0);
  if (e != cudaSuccess) return e;
  set_kernel_info("patch_pack_kernel %s C=%d T=%d H=%d W=%d patch=1x2x2", unpack ? "unpack" : "pack", C, T, H, W);
  return cudaGetLastError();
}

cudaError_t launch_input_proj(const InputProjArgs& a, cudaStream_t st) {
  const int smem = 2 * a.K * IP_ROWS * (int)sizeof(float);
  cudaError_t e = cudaFuncSetAttribute(input_proj_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const dim3 grid((unsigned)((a.n + IP_ROWS - 1) / IP_ROWS), (unsigned)((a.D + IP_COLS - 1) / IP_COLS));
  e = launch_kernel(input_proj_kernel, grid, dim3(IP_THREADS), (size_t)smem, st, a);
  if (e != cudaSuccess) return e;
  set_kernel_info("input_proj_kernel fp32 tile=%dx%d k=%d reg-tile=8x8 rows=%d", IP_ROWS, IP_COLS, a.K, a.n);
  return cudaGetLastError();
}

cudaError_t launch_index_copy(int n, int D, const __nv_bfloat16* src, const int32_t* dst, int n_dst,
                              __nv_bfloat16* out, uint32_t* err, cudaStream_t st) {
  cudaError_t e = launch_kernel(index_copy_kernel, dim3(grid_for((long long)n * 32, 256, 8)), dim3(256), 0, st, n,
                                D, src, dst, n_dst, out, err);
  if (e != cudaSuccess) return e;
  set_kernel_info("index_copy_kernel warp-per-row rows=%d", n);
  return cudaGetLastError();
}

cudaError_t launch_sinusoid(int T, const float* t, float* e_out, cudaStream_t st) {
  cudaError_t e = launch_kernel(sinusoid_kernel, dim3((T * 128 + 255) / 256), dim3(256), 0, st, T, t, e_out);
  if (e != cudaSuccess) return e;
  set_kernel_info("sinusoid_kernel fp32 T=%d width=256", T);
  return cudaGetLastError();
}

cudaError_t launch_rows_linear(int T, int K, int N, const float* in, const float* w, const float* b, int act,
                               float* out, cudaStream_t st) {
  cudaError_t e = launch_kernel(rows_linear_kernel, dim3(grid_for((long long)N * 32, 256, 8)), dim3(256), 0, st, T,
                                K, N, in, w, b, act, out);
  if (e != cudaSuccess) return e;
  set_kernel_info("rows_linear_kernel fp32 warp-per-column T=%d K=%d N=%d act=%d", T, K, N, act);
  return cudaGetLastError();
}

}  // namespace h3
