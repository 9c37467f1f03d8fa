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
// channels").  One warp per (row, head): lane l holds channels 4l..4l+3; lanes
// 0-11 hold the first half of the 96 rotary channels and exchange with lanes
// 12-23, which hold the partners j+48; lanes 24-31 hold the 32 pass-through
// channels.
#include "h3_device.cuh"
#include "h3_internal.h"

namespace h3 {

namespace {
constexpr int MOD_THREADS = 256;
constexpr int MOD_MAXC = 4;  // 16-byte chunks per thread: D <= 256 * 4 * 8 = 8192
}  // namespace

__global__ void __launch_bounds__(MOD_THREADS) modulate_kernel(const ModulateArgs a) {
  const int row = blockIdx.x;
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
  modulate_kernel<<<a.S, MOD_THREADS, 0, stream>>>(a);
  set_kernel_info("modulate_kernel rows=%d threads=%d vec=16B reduce=fixed-tree", a.S, MOD_THREADS);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) rope_qknorm_kernel(const RopeArgs a) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long gw = (long long)blockIdx.x * 8 + warp;
  if (gw >= (long long)a.S * a.H) return;
  const int i = (int)(gw / a.H), h = (int)(gw % a.H);
  float pos[3];
  bool valid = true;
#pragma unroll
  for (int ax = 0; ax < 3; ++ax) {
    const int p = a.pos[(size_t)i * 3 + ax];
    if ((unsigned)p >= (1u << 24)) valid = false;
    pos[ax] = (float)p;
  }
  if (!valid) {
    if (lane == 0) record_error(a.err, DEVERR_INDEX);
    return;
  }
  // angles of this lane's four channels (lanes 0-23; both partners compute
  // the same j = 4*(lane mod 12) + e)
  float cs[4], sn[4];
  const int jl = (lane < 12 ? lane : lane - 12) * 4;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const int j = jl + e;
    const int band = j >> 4;
    const float p = band == 0 ? pos[0] : (band == 1 ? pos[1] : pos[2]);
    sincosf(p * a.omega[j & 15], &sn[e], &cs[e]);
  }
  const int partner = lane < 12 ? lane + 12 : (lane < 24 ? lane - 12 : lane);
#pragma unroll
  for (int part = 0; part < 2; ++part) {
    __nv_bfloat16* base = (part ? a.k : a.q) + (size_t)i * a.row_stride + (size_t)h * a.head_stride;
    const __nv_bfloat16* gain = part ? a.k_gain : a.q_gain;
    uint2 raw = *reinterpret_cast<const uint2*>(base + lane * 4);
    float v[4] = {bf16_lo(raw.x), bf16_hi(raw.x), bf16_lo(raw.y), bf16_hi(raw.y)};
    float ss = 0.0f;
#pragma unroll
    for (int e = 0; e < 4; ++e) ss = __fmaf_rn(v[e], v[e], ss);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    const float inv = 1.0f / sqrtf(ss * (1.0f / 128.0f) + a.eps);
    float n[4], out[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) n[e] = bf16_round((v[e] * inv) * __bfloat162float(gain[lane * 4 + e]));
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float other = __shfl_sync(0xffffffffu, n[e], partner);
      if (lane < 12) out[e] = __fmaf_rn(n[e], cs[e], -(other * sn[e]));
      else if (lane < 24) out[e] = __fmaf_rn(n[e], cs[e], other * sn[e]);
      else out[e] = n[e];
    }
    raw.x = pack_bf16x2(out[0], out[1]);
    raw.y = pack_bf16x2(out[2], out[3]);
    *reinterpret_cast<uint2*>(base + lane * 4) = raw;
  }
}

cudaError_t launch_rope_qknorm(const RopeArgs& a, cudaStream_t stream) {
  const long long warps = (long long)a.S * a.H;
  const unsigned blocks = (unsigned)((warps + 7) / 8);
  rope_qknorm_kernel<<<blocks, 256, 0, stream>>>(a);
  set_kernel_info("rope_qknorm_kernel warp-per-(row,head) rows=%d heads=%d", a.S, a.H);
  return cudaGetLastError();
}

}  // namespace h3
