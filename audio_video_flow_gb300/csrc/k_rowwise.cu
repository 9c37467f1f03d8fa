// Row-wise, HBM-bound kernels of the H3 block.
//
// modulate_kernel: RMSNorm + AdaLN modulation of one branch (RFC section 2,
// fingerprint row "Block norm", eps 1e-5; section 5 adaln_row_gather:
// row = timestep_index*3 + token_tag).  One CTA per packed row: the row is
// read once with 16-byte loads into registers, its sum of squares reduced in a
// fixed order (per-thread chunks, warp butterfly, then the 8 warps in order),
// and the modulated row written once.  The six-chunk table rows are shared by
// all rows with the same (timestep, tag) and stay in L2.
//
// rope_qknorm_kernel: standalone per-head Q/K RMSNorm + partial three-axis
// MM-RoPE, in place (RFC section 2 rows "Q/K preprocessing", "Rotary
// channels"); layout described at the kernel.
#include "h3_device.cuh"
#include "h3_internal.h"

namespace h3 {

namespace {
constexpr int MOD_THREADS = 256;
constexpr int MOD_MAXC = 4;  // 16-byte chunks per thread: D <= 256 * 4 * 8 = 8192
}  // namespace

__global__ void __launch_bounds__(MOD_THREADS) modulate_kernel(const ModulateArgs a) {
  const int row = blockIdx.x;
  griddep_launch_dependents();
  griddep_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __shared__ float red[MOD_THREADS / 32];
  const int tg = a.tag[row], ti = a.tidx[row];
  if ((unsigned)tg > 2u || (unsigned)ti >= (unsigned)a.T) {
    if (threadIdx.x == 0) record_error(a.err, DEVERR_INDEX);
    return;
  }
  const int nch = a.D >> 3;
  const uint4* xr = reinterpret_cast<const uint4*>(a.x + (size_t)row * a.D);
  uint4 xv[MOD_MAXC];
  float ss = 0.0f;
#pragma unroll
  for (int i = 0; i < MOD_MAXC; ++i) {
    const int c = threadIdx.x + i * MOD_THREADS;
    if (c < nch) {
      xv[i] = xr[c];
      const uint32_t w[4] = {xv[i].x, xv[i].y, xv[i].z, xv[i].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float lo = bf16_lo(w[e]), hi = bf16_hi(w[e]);
        ss = __fmaf_rn(lo, lo, ss);
        ss = __fmaf_rn(hi, hi, ss);
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if (lane == 0) red[warp] = ss;
  __syncthreads();
  float tot = 0.0f;
#pragma unroll
  for (int w = 0; w < MOD_THREADS / 32; ++w) tot += red[w];
  const float inv = 1.0f / sqrtf(tot / (float)a.D + a.eps);

  const __nv_bfloat16* trow = a.table + (size_t)(ti * 3 + tg) * 6 * a.D;
  const uint4* shp = reinterpret_cast<const uint4*>(trow + (size_t)a.chunk_shift * a.D);
  const uint4* scp = reinterpret_cast<const uint4*>(trow + (size_t)a.chunk_scale * a.D);
  const uint4* gp = reinterpret_cast<const uint4*>(a.gain);
  uint4* hp = reinterpret_cast<uint4*>(a.h + (size_t)row * a.D);
#pragma unroll
  for (int i = 0; i < MOD_MAXC; ++i) {
    const int c = threadIdx.x + i * MOD_THREADS;
    if (c < nch) {
      const uint4 gv = gp[c], shv = shp[c], scv = scp[c];
      const uint32_t xw[4] = {xv[i].x, xv[i].y, xv[i].z, xv[i].w};
      const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w};
      const uint32_t hw[4] = {shv.x, shv.y, shv.z, shv.w};
      const uint32_t cw[4] = {scv.x, scv.y, scv.z, scv.w};
      uint32_t ow[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float nlo = (bf16_lo(xw[e]) * inv) * bf16_lo(gw[e]);
        const float nhi = (bf16_hi(xw[e]) * inv) * bf16_hi(gw[e]);
        const float ylo = __fmaf_rn(nlo, 1.0f + bf16_lo(cw[e]), bf16_lo(hw[e]));
        const float yhi = __fmaf_rn(nhi, 1.0f + bf16_hi(cw[e]), bf16_hi(hw[e]));
        ow[e] = pack_bf16x2(ylo, yhi);
      }
      hp[c] = make_uint4(ow[0], ow[1], ow[2], ow[3]);
    }
  }
}

cudaError_t launch_modulate(const ModulateArgs& a, cudaStream_t stream) {
  cudaError_t e = launch_kernel(modulate_kernel, dim3(a.S), dim3(MOD_THREADS), 0, stream, a);
  if (e != cudaSuccess) return e;
  set_kernel_info("modulate_kernel rows=%d threads=%d vec=16B reduce=fixed-tree", a.S, MOD_THREADS);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// One CTA per packed row.  The row's 48 rotation angles (bands t, h, w x 16
// frequencies, fp32(pos) * omega_f in fp32) are computed once into shared
// memory; then each warp takes whole heads: lanes 0-15 hold q, lanes 16-31
// hold k, lane l of a half owning channels 8l..8l+7 (16-byte accesses).  The
// rotation pairs channel j < 48 with j + 48, i.e. half-lane l < 6 with l + 6;
// half-lanes 12-15 carry the 32 pass-through channels.  A warp issues the
// loads of all its heads (up to 8 x 512 bytes) before it computes.
__global__ void __launch_bounds__(256) rope_qknorm_kernel(const RopeArgs a) {
  const int i = blockIdx.x;
  griddep_launch_dependents();
  griddep_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int hl = lane & 15;                 // lane within the q or k half
  const bool is_k = lane >= 16;
  __shared__ float s_cos[48], s_sin[48];
  __shared__ int s_bad;
  // heads warp, warp + 8, ...: issue this warp's loads first (up to 8 x 512
  // bytes), so their latency overlaps the angle set-up below
  constexpr int kMaxHeadsPerWarp = 8;   // H <= 64 per pass
  __nv_bfloat16* base = (is_k ? a.k : a.q) + (size_t)i * a.row_stride + hl * 8;
  uint4 r[kMaxHeadsPerWarp];
#pragma unroll
  for (int u = 0; u < kMaxHeadsPerWarp; ++u) {
    const int h = warp + 8 * u;
    if (h < a.H) r[u] = *reinterpret_cast<const uint4*>(base + (size_t)h * a.head_stride);
  }
  if (threadIdx.x == 0) s_bad = 0;
  __syncthreads();
  if (threadIdx.x < 48) {
    const int band = threadIdx.x >> 4, f = threadIdx.x & 15;
    const int p = a.pos[(size_t)i * 3 + band];
    if ((unsigned)p >= (1u << 24)) s_bad = 1;
    float sn, cs;
    sincosf((float)p * a.omega[f], &sn, &cs);
    s_cos[threadIdx.x] = cs;
    s_sin[threadIdx.x] = sn;
  }
  __syncthreads();
  if (s_bad) {
    if (threadIdx.x == 0) record_error(a.err, DEVERR_INDEX);
    return;
  }
  const int partner = hl < 6 ? lane + 6 : (hl < 12 ? lane - 6 : lane);
  float cs[8], sn[8], g[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const int j = (hl < 12 ? (hl % 6) : 0) * 8 + e;   // rotation column of this channel
    cs[e] = s_cos[j];
    sn[e] = s_sin[j];
    g[e] = __bfloat162float((is_k ? a.k_gain : a.q_gain)[hl * 8 + e]);
  }
  for (int hb = 0; hb < a.H; hb += 8 * kMaxHeadsPerWarp) {
    if (hb > 0) {
#pragma unroll
      for (int u = 0; u < kMaxHeadsPerWarp; ++u) {
        const int h = hb + warp + 8 * u;
        if (h < a.H) r[u] = *reinterpret_cast<const uint4*>(base + (size_t)h * a.head_stride);
      }
    }
#pragma unroll
    for (int u = 0; u < kMaxHeadsPerWarp; ++u) {
      const int h = hb + warp + 8 * u;
      if (h >= a.H) break;
      const uint32_t w[4] = {r[u].x, r[u].y, r[u].z, r[u].w};
      float v[8];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        v[2 * e] = bf16_lo(w[e]);
        v[2 * e + 1] = bf16_hi(w[e]);
      }
      float ss = 0.0f;
#pragma unroll
      for (int e = 0; e < 8; ++e) ss = __fmaf_rn(v[e], v[e], ss);
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);   // within the half
      const float inv = 1.0f / sqrtf(ss * (1.0f / 128.0f) + a.eps);
      float n[8], out[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) n[e] = bf16_round((v[e] * inv) * g[e]);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float other = __shfl_sync(0xffffffffu, n[e], partner);
        if (hl < 6) out[e] = __fmaf_rn(n[e], cs[e], -(other * sn[e]));
        else if (hl < 12) out[e] = __fmaf_rn(n[e], cs[e], other * sn[e]);
        else out[e] = n[e];
      }
      *reinterpret_cast<uint4*>(base + (size_t)h * a.head_stride) =
          make_uint4(pack_bf16x2(out[0], out[1]), pack_bf16x2(out[2], out[3]), pack_bf16x2(out[4], out[5]),
                     pack_bf16x2(out[6], out[7]));
    }
  }
}

cudaError_t launch_rope_qknorm(const RopeArgs& a, cudaStream_t stream) {
  cudaError_t e = launch_kernel(rope_qknorm_kernel, dim3(a.S), dim3(256), 0, stream, a);
  if (e != cudaSuccess) return e;
  set_kernel_info("rope_qknorm_kernel cta-per-row angles-in-smem vec=16B rows=%d heads=%d", a.S, a.H);
  return cudaGetLastError();
}

}  // namespace h3
