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
// final AdaLN table: out[t][j] = SiLU(t_cond[t]) . w[j] + b[j], fp32, j < 2D,
// for one or more tables (the modalities) in one launch: weight row j of
// table m is work unit m * 2D + j, so the modalities stream back to back
// without a second launch's ramp.  Three CTAs per SM, each holding u = SiLU(t_cond) [T][C] in shared memory.
// A warp owns one weight row at a time and issues the 16-byte loads of half
// the row before it multiplies (lane l takes float4 columns l + 32i, at most
// 11 per lane and half for C <= 2816), so each resident warp keeps half a
// row (up to 5.5 KB) in flight; the lane's T running sums go on in column
// order across the halves and are reduced over the warp with a fixed xor
// tree.  Three CTAs of 256 threads fit in the registers with half rows (two
// for T > 8): the
// 10,752 rows of an H3 modality then take three rounds of the 3648 resident
// warps (two CTAs and whole rows took five, the last 42 % full).  The
// kernel is bound by the 2D x C fp32 weights streamed once.
// ---------------------------------------------------------------------------
constexpr int FA_THREADS = 256;
constexpr int FA_MAX_LOADS = kMaxCondDim / 4 / 32;   // float4 loads per lane per row
constexpr int FA_HALF_LOADS = FA_MAX_LOADS / 2;        // per half row
// resident CTAs per SM: three, or two for the 16 running sums of T > 8
// (which would not fit three CTAs' registers without spilling)
__host__ __device__ constexpr int fa_ctas_per_sm(int TT) { return TT >= 16 ? 2 : 3; }
static_assert(FA_MAX_LOADS * 4 * 32 == kMaxCondDim, "a lane's share of the widest row is whole float4s");
static_assert(FA_HALF_LOADS * 2 == FA_MAX_LOADS, "the row splits into two equal halves");

// TT: timestep rows rounded up to a power of two (the unrolled sum loops
// cover TT rows, so T = 1 compiles to one sum per lane)
template <int TT>
__global__ void __launch_bounds__(FA_THREADS, fa_ctas_per_sm(TT)) final_adaln_kernel(const __grid_constant__ FinalAdalnArgs a) {
  extern __shared__ float u[];   // [T][C]
  griddep_launch_dependents();
  griddep_wait();
  const int T = a.T, C = a.C, rows = a.rows;
  for (int i = threadIdx.x; i < T * C; i += blockDim.x) {
    const float x = a.t_cond[i];
    u[i] = x / (1.0f + expf(-x));
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nw = blockDim.x >> 5;
  const int c4 = C >> 2;
  for (int jm = blockIdx.x * nw + warp; jm < a.n_tables * rows; jm += gridDim.x * nw) {
    const int m = jm / rows, j = jm - m * rows;   // table m, weight row j
    const float* __restrict__ b = a.b[m];
    float* __restrict__ out = a.out[m];
    const float4* wr = reinterpret_cast<const float4*>(a.w[m] + (size_t)j * C);
    float acc[TT];
#pragma unroll
    for (int t = 0; t < TT; ++t) acc[t] = 0.0f;
    // the row in two halves (each lane's loads of a half in flight together),
    // the sums running on in column order across them
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      float4 wv[FA_HALF_LOADS];
#pragma unroll
      for (int q = 0; q < FA_HALF_LOADS; ++q) {
        const int kk = lane + (h * FA_HALF_LOADS + q) * 32;
        wv[q] = kk < c4 ? __ldcs(wr + kk) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int q = 0; q < FA_HALF_LOADS; ++q) {
        const int kk = lane + (h * FA_HALF_LOADS + q) * 32;
        if (kk < c4) {
#pragma unroll
          for (int t = 0; t < TT; ++t) {
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
    for (int t = 0; t < TT; ++t) {
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
// Velocity head.  A cluster of KS CTAs (KS in {1, 2, 4, 8, 16}: the fewest
// that give two CTAs per SM, else 16 where the device runs clusters of 16,
// else 8) takes 96 selected rows and all P columns (P
// padded to 16 * PT, PT in {2, 4, 6, 8}); CTA rank ks of the cluster owns the
// ks-th of KS contiguous ranges of the reduction axis D (whole 32-column
// chunks).  The 14,580 video rows of an evaluation make 152 tiles in pairs:
// 304 CTAs, one wave at two per SM.
//   1. Each CTA sums the squares of its range of each row (lane partials in
//      column order, fixed xor tree); with KS > 1, after a cluster barrier,
//      every CTA adds the KS partials in rank order; inv = 1/sqrt(ss/D + eps).
//   2. Each CTA walks its range in 32-column chunks: the modulated
//      activations a[k][row] = (x * inv) * (1 + scale) + shift and the head
//      chunk w[k][p] are staged in shared memory (double-buffered; the next
//      chunk's 16-byte global loads are in flight during the products), and
//      thread (ty, tx) accumulates an 8-row x PT-column register tile in k
//      order, reading its 8 rows with two 16-byte and its PT columns with
//      8-byte shared loads per k.
//   3. With KS = 1 each thread adds the bias and writes its tile.  Otherwise
//      the partial tiles are left in shared memory; after a cluster barrier
//      rank ks adds, for its 96 / KS rows of the tile, the KS partials in
//      rank order over distributed shared memory, adds the bias and writes
//      the rows.
// For a given row count every output is one fixed-order fp32 sum.
// Rows whose metadata is out of range are reported and left unwritten.
// ---------------------------------------------------------------------------
constexpr int OH_ROWS = 96, OH_KC = 32, OH_THREADS = 192, OH_MAX_KS = 16;
static_assert(OH_ROWS == 8 * (OH_THREADS / 16), "16 column groups x 8-row groups cover the tile");
static_assert(OH_THREADS == 2 * OH_ROWS, "two staging threads per row");
static_assert(OH_ROWS % OH_MAX_KS == 0, "every k-split divides the rows");
constexpr int OH_TSLOTS = (16 * 2 * (OH_KC / 4) + OH_THREADS - 1) / OH_THREADS;   // table float4 per thread

template <int PT>
struct OhCfg {
  static constexpr int PW = 16 * PT;                    // padded head width
  static constexpr int WS = PW + 2;                     // s_w row stride (even, 2 mod 32)
  static constexpr int A_FLOATS = OH_KC * OH_ROWS;      // one s_a buffer
  static constexpr int W_FLOATS = OH_KC * WS;           // one s_w buffer
  static constexpr int STAGE_FLOATS = 2 * (A_FLOATS + W_FLOATS);
  static constexpr int TILE_FLOATS = OH_ROWS * PW;      // partial tile for the cluster reduction
  static constexpr int FLOATS = STAGE_FLOATS > TILE_FLOATS ? STAGE_FLOATS : TILE_FLOATS;
  static constexpr int SMEM = FLOATS * 4;
  static constexpr int WSLOTS = (PW * (OH_KC / 4) + OH_THREADS - 1) / OH_THREADS;   // float4 per thread
};

__device__ __forceinline__ float ld_shared_cluster_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}

template <int PT>
__global__ void __launch_bounds__(OH_THREADS, 2) output_head_kernel(const OutputHeadArgs a) {
  using Cf = OhCfg<PT>;
  constexpr int PW = Cf::PW, WS = Cf::WS;
  extern __shared__ __align__(16) float oh_smem[];
  float* s_a = oh_smem;                          // [2][OH_KC][OH_ROWS]
  float* s_w = oh_smem + 2 * Cf::A_FLOATS;       // [2][OH_KC][WS]
  float* s_tile = oh_smem;                       // [OH_ROWS][PW] after the main loop
  __shared__ float s_ss[OH_ROWS];                // this CTA's partial sums of squares
  __shared__ __align__(16) float s_tab[2][16][2][OH_KC];   // shift / scale slices per timestep row
  __shared__ float s_inv[OH_ROWS];
  __shared__ int s_row[OH_ROWS], s_t[OH_ROWS];
  griddep_launch_dependents();
  griddep_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int KS = (int)cluster_nctarank();
  const int ks = (int)cluster_ctarank();
  const int i0 = (blockIdx.x / KS) * OH_ROWS;
  const int D = a.D, P = a.P;
  const int nch = D / OH_KC;
  const int c_lo = (ks * nch) / KS, c_hi = ((ks + 1) * nch) / KS;   // chunks of this CTA
  const int k_lo = c_lo * OH_KC, k_hi = c_hi * OH_KC;
  if (threadIdx.x < OH_ROWS) {
    const int i = i0 + (int)threadIdx.x;
    int r = -1, t = 0;
    if (i < a.n_sel) {
      r = a.rows[i];
      if ((unsigned)r >= (unsigned)a.S) {
        if (ks == 0) record_error(a.err, DEVERR_INDEX);
        r = -1;
      } else {
        t = a.tidx[r];
        if ((unsigned)t >= (unsigned)a.T) {
          if (ks == 0) record_error(a.err, DEVERR_INDEX);
          r = -1;
          t = 0;
        }
      }
    }
    s_row[threadIdx.x] = r;
    s_t[threadIdx.x] = t;
  }
  __syncthreads();
  // 1. partial sums of squares over [k_lo, k_hi), sixteen rows per warp
  for (int rr = warp; rr < OH_ROWS; rr += OH_THREADS / 32) {
    const int r = s_row[rr];
    float ss = 0.0f;
    if (r >= 0) {
      const uint4* xr = reinterpret_cast<const uint4*>(a.x + (size_t)r * D + k_lo);
      for (int c = lane; c < ((k_hi - k_lo) >> 3); c += 32) {
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
    if (lane == 0) s_ss[rr] = ss;
  }
  if (KS > 1) {
    cluster_sync();
    if (threadIdx.x < OH_ROWS) {
      const uint32_t my = smem_u32(&s_ss[threadIdx.x]);
      float ss = 0.0f;
      for (int q = 0; q < KS; ++q) ss += ld_shared_cluster_f32(mapa_shared(my, (uint32_t)q));
      s_inv[threadIdx.x] = 1.0f / sqrtf(ss / (float)D + a.eps);
    }
  } else {
    __syncthreads();
    if (threadIdx.x < OH_ROWS) s_inv[threadIdx.x] = 1.0f / sqrtf(s_ss[threadIdx.x] / (float)D + a.eps);
  }
  __syncthreads();

  // 2. staging roles.  activations: row ar = tid / 2, columns ak..ak+15 of the
  // chunk; head: float4 slots f = tid + 192 e over PW rows x 8 float4 (rows >= P
  // are zero)
  const int ar = threadIdx.x >> 1, ak = (threadIdx.x & 1) * 16;
  const int my_row = s_row[ar];
  const float my_inv = s_inv[ar];
  const int my_t = s_t[ar];
  constexpr int WSLOTS = Cf::WSLOTS;
  // the table slice [T][shift, scale][32 columns] of a chunk: float4 slots
  // f = tid + 192 e over 16 timestep rows x 2 x 8, loaded two chunks ahead
  auto load_tab = [&](int k0, float4 (&tv)[OH_TSLOTS]) {
#pragma unroll
    for (int e = 0; e < OH_TSLOTS; ++e) {
      const int f = (int)threadIdx.x + e * OH_THREADS;
      const int tb_t = f >> 4, tb_h = (f >> 3) & 1, tb_q = f & 7;
      tv[e] = tb_t < a.T ? *reinterpret_cast<const float4*>(a.table + ((size_t)tb_t * 2 + tb_h) * D + k0 + tb_q * 4)
                         : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  };
  auto put_tab = [&](int tbuf, const float4 (&tv)[OH_TSLOTS]) {
#pragma unroll
    for (int e = 0; e < OH_TSLOTS; ++e) {
      const int f = (int)threadIdx.x + e * OH_THREADS;
      const int tb_t = f >> 4, tb_h = (f >> 3) & 1, tb_q = f & 7;
      if (tb_t < a.T) *reinterpret_cast<float4*>(&s_tab[tbuf][tb_t][tb_h][tb_q * 4]) = tv[e];
    }
  };
  auto load_chunk = [&](int k0, uint4 (&xv)[2], float4 (&wv)[WSLOTS]) {
    if (my_row >= 0) {
      const uint4* xp = reinterpret_cast<const uint4*>(a.x + (size_t)my_row * D + k0 + ak);
      xv[0] = xp[0];
      xv[1] = xp[1];
    }
#pragma unroll
    for (int e = 0; e < WSLOTS; ++e) {
      const int f = (int)threadIdx.x + e * OH_THREADS;
      const int p = f / (OH_KC / 4), kq = f % (OH_KC / 4);
      wv[e] = (p < P) ? *reinterpret_cast<const float4*>(a.w + (size_t)p * D + k0 + kq * 4)
                      : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  };
  auto store_chunk = [&](int buf, const uint4 (&xv)[2], const float4 (&wv)[WSLOTS]) {
    float* sa = s_a + buf * Cf::A_FLOATS;
    float* sw = s_w + buf * Cf::W_FLOATS;
    const uint32_t xw[8] = {xv[0].x, xv[0].y, xv[0].z, xv[0].w, xv[1].x, xv[1].y, xv[1].z, xv[1].w};
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      float4 sh = make_float4(0.f, 0.f, 0.f, 0.f), sc = sh;
      if (my_row >= 0) {
        sh = *reinterpret_cast<const float4*>(&s_tab[buf][my_t][0][ak + 4 * g]);
        sc = *reinterpret_cast<const float4*>(&s_tab[buf][my_t][1][ak + 4 * g]);
      }
      const float shv[4] = {sh.x, sh.y, sh.z, sh.w};
      const float scv[4] = {sc.x, sc.y, sc.z, sc.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int c = 4 * g + e;
        float val = 0.0f;
        if (my_row >= 0) {
          const float xvv = (c & 1) ? bf16_hi(xw[c >> 1]) : bf16_lo(xw[c >> 1]);
          val = __fmaf_rn(xvv * my_inv, 1.0f + scv[e], shv[e]);
        }
        sa[(ak + c) * OH_ROWS + ar] = val;
      }
    }
#pragma unroll
    for (int e = 0; e < WSLOTS; ++e) {
      const int f = (int)threadIdx.x + e * OH_THREADS;
      const int p = f / (OH_KC / 4), kq = f % (OH_KC / 4);
      if (p < PW) {
        sw[(kq * 4 + 0) * WS + p] = wv[e].x;
        sw[(kq * 4 + 1) * WS + p] = wv[e].y;
        sw[(kq * 4 + 2) * WS + p] = wv[e].z;
        sw[(kq * 4 + 3) * WS + p] = wv[e].w;
      }
    }
  };

  const int ty = threadIdx.x >> 4, tx = threadIdx.x & 15;   // rows 8ty..8ty+7, columns PT tx..PT tx+PT-1
  float acc[8][PT];
#pragma unroll
  for (int r8 = 0; r8 < 8; ++r8)
#pragma unroll
    for (int c = 0; c < PT; ++c) acc[r8][c] = 0.0f;
  uint4 xv[2] = {make_uint4(0u, 0u, 0u, 0u), make_uint4(0u, 0u, 0u, 0u)};
  float4 wv[WSLOTS];
  float4 tv[OH_TSLOTS];
  if (k_lo < k_hi) {
    load_tab(k_lo, tv);
    put_tab(0, tv);
  }
  if (k_lo + OH_KC < k_hi) {
    load_tab(k_lo + OH_KC, tv);
    put_tab(1, tv);
  }
  __syncthreads();
  if (k_lo < k_hi) {
    load_chunk(k_lo, xv, wv);
    store_chunk(0, xv, wv);
  }
  __syncthreads();
  int buf = 0;
  for (int k0 = k_lo; k0 < k_hi; k0 += OH_KC) {
    const bool more = k0 + OH_KC < k_hi;
    const bool more2 = k0 + 2 * OH_KC < k_hi;
    if (more) load_chunk(k0 + OH_KC, xv, wv);   // in flight during the products
    if (more2) load_tab(k0 + 2 * OH_KC, tv);
    const float* sa = s_a + buf * Cf::A_FLOATS;
    const float* sw = s_w + buf * Cf::W_FLOATS;
#pragma unroll 2
    for (int kk = 0; kk < OH_KC; ++kk) {
      const float4 a0 = *reinterpret_cast<const float4*>(&sa[kk * OH_ROWS + ty * 8]);
      const float4 a1 = *reinterpret_cast<const float4*>(&sa[kk * OH_ROWS + ty * 8 + 4]);
      float w[PT];
#pragma unroll
      for (int m = 0; m < PT / 2; ++m) {
        const float2 w2 = *reinterpret_cast<const float2*>(&sw[kk * WS + tx * PT + 2 * m]);
        w[2 * m] = w2.x;
        w[2 * m + 1] = w2.y;
      }
      const float a8[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
#pragma unroll
      for (int r8 = 0; r8 < 8; ++r8)
#pragma unroll
        for (int c = 0; c < PT; ++c) acc[r8][c] = __fmaf_rn(a8[r8], w[c], acc[r8][c]);
    }
    if (more) store_chunk(buf ^ 1, xv, wv);
    // the table slice two chunks ahead goes where this chunk's was (last
    // read by the staging before the previous barrier)
    if (more2) put_tab(buf, tv);
    __syncthreads();
    buf ^= 1;
  }

  // 3. the tile: straight out with KS = 1, else partial tiles to shared
  // memory and rank ks reduces its 96 / KS rows over the cluster
  if (KS == 1) {
#pragma unroll
    for (int r8 = 0; r8 < 8; ++r8) {
      const int rr = ty * 8 + r8, i = i0 + rr;
      if (s_row[rr] < 0 || i >= a.n_sel) continue;
#pragma unroll
      for (int c = 0; c < PT; ++c) {
        const int p = tx * PT + c;
        if (p < P) a.out[(size_t)i * P + p] = acc[r8][c] + (a.b ? a.b[p] : 0.0f);
      }
    }
    return;
  }
#pragma unroll
  for (int r8 = 0; r8 < 8; ++r8)
#pragma unroll
    for (int c = 0; c < PT; ++c) s_tile[(ty * 8 + r8) * PW + tx * PT + c] = acc[r8][c];
  cluster_sync();
  const int slice = OH_ROWS / KS;
  for (int e = (int)threadIdx.x; e < slice * PW; e += OH_THREADS) {
    const int rr = ks * slice + e / PW, p = e % PW;
    if (p >= P) continue;
    const uint32_t my = smem_u32(&s_tile[rr * PW + p]);
    float v = 0.0f;
    for (int q = 0; q < KS; ++q) v += ld_shared_cluster_f32(mapa_shared(my, (uint32_t)q));
    const int i = i0 + rr;
    if (s_row[rr] >= 0 && i < a.n_sel) a.out[(size_t)i * P + p] = v + (a.b ? a.b[p] : 0.0f);
  }
  cluster_sync();   // no CTA leaves while another still reads its shared memory
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

template <int TT>
static cudaError_t launch_fa(const FinalAdalnArgs& a, int& grid, cudaStream_t st) {
  const int smem = a.T * a.C * (int)sizeof(float);
  const int warps = FA_THREADS / 32;
  const long long units = (long long)a.n_tables * a.rows;
  grid = (int)((units + warps - 1) / warps);
  const int cap = fa_ctas_per_sm(TT) * num_sms();   // resident CTAs; warps loop over rows
  if (grid > cap) grid = cap;
  cudaError_t e = cudaFuncSetAttribute(final_adaln_kernel<TT>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  return launch_kernel(final_adaln_kernel<TT>, dim3(grid), dim3(FA_THREADS), (size_t)smem, st, a);
}

cudaError_t launch_final_adaln(const FinalAdalnArgs& a, cudaStream_t st) {
  int grid = 0;
  cudaError_t e;
  if (a.T <= 1) e = launch_fa<1>(a, grid, st);
  else if (a.T <= 2) e = launch_fa<2>(a, grid, st);
  else if (a.T <= 4) e = launch_fa<4>(a, grid, st);
  else if (a.T <= 8) e = launch_fa<8>(a, grid, st);
  else e = launch_fa<16>(a, grid, st);
  if (e != cudaSuccess) return e;
  set_kernel_info("final_adaln_kernel fp32 warp-per-row half-rows-in-flight tables=%d T=%d C=%d rows=%d grid=%d",
                  a.n_tables, a.T, a.C, a.rows, grid);
  return cudaGetLastError();
}

// The k-split: the fewest of 1, 2, 4, 8 CTAs per 96-row tile that give two
// CTAs per SM; when none does, 16 (a cluster size beyond the portable 8,
// taken only where the device can hold such a cluster of this kernel), else
// 8.  A short selection such as the 1024 audio rows (11 tiles) then walks 10
// or 11 chunks of 32 columns per CTA instead of 21: its chunks are short, so
// each waits for its global loads, and the time follows the chunk count.
template <int PT>
static cudaError_t launch_head(const OutputHeadArgs& a, int tiles, int& ks, cudaStream_t st) {
  constexpr int smem = OhCfg<PT>::SMEM;
  cudaError_t e = cudaFuncSetAttribute(output_head_kernel<PT>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int target = 2 * num_sms();
  ks = 0;
  for (int k : {1, 2, 4, 8})
    if (ks == 0 && (long long)tiles * k >= target) ks = k;
  if (ks == 0) {
    ks = 8;
    if (cudaFuncSetAttribute(output_head_kernel<PT>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) ==
        cudaSuccess) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3((unsigned)(tiles * OH_MAX_KS));
      cfg.blockDim = dim3(OH_THREADS);
      cfg.dynamicSmemBytes = smem;
      cfg.stream = st;
      cudaLaunchAttribute attr;
      attr.id = cudaLaunchAttributeClusterDimension;
      attr.val.clusterDim.x = OH_MAX_KS;
      attr.val.clusterDim.y = 1;
      attr.val.clusterDim.z = 1;
      cfg.attrs = &attr;
      cfg.numAttrs = 1;
      int clusters = 0;
      if (cudaOccupancyMaxActiveClusters(&clusters, output_head_kernel<PT>, &cfg) == cudaSuccess && clusters >= 1)
        ks = OH_MAX_KS;
      else
        (void)cudaGetLastError();   // the query's error is not this launch's
    } else {
      (void)cudaGetLastError();
    }
  }
  return launch_kernel_cluster(output_head_kernel<PT>, dim3(tiles * ks), dim3(OH_THREADS), smem, st, ks, a);
}

cudaError_t launch_output_head(const OutputHeadArgs& a, cudaStream_t st) {
  const int tiles = (a.n_sel + OH_ROWS - 1) / OH_ROWS;
  int ks = 0;
  const int pt = a.P <= 32 ? 2 : (a.P <= 64 ? 4 : (a.P <= 96 ? 6 : 8));
  cudaError_t e;
  switch (pt) {
    case 2: e = launch_head<2>(a, tiles, ks, st); break;
    case 4: e = launch_head<4>(a, tiles, ks, st); break;
    case 6: e = launch_head<6>(a, tiles, ks, st); break;
    default: e = launch_head<8>(a, tiles, ks, st); break;
  }
  if (e != cudaSuccess) return e;
  set_kernel_info("output_head_kernel<%d> fp32 rows/tile=%d k-split=%d (cluster, rank-order sums) k_chunk=%d "
                  "reg-tile=8x%d P=%d rows=%d", pt, OH_ROWS, ks, OH_KC, pt, a.P, a.n_sel);
  return cudaGetLastError();
}

}  // namespace h3
