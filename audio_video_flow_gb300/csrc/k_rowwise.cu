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
// channels"); a persistent TMA-fed kernel, structure described at the kernel.
#include "h3_device.cuh"
#include "h3_internal.h"

namespace h3 {

namespace {
// The row's sum of squares follows one fixed tree whatever the CTA size: 256
// virtual threads, virtual thread vt summing 16-byte chunks vt, vt + 256, ...
// in order, a butterfly over each 32 virtual threads, then the eight warp
// sums in order.  A CTA runs it with 256 threads (V = 1) for short documents,
// where each row's latency matters most (505 rows: 8.6 us against 10.5 with
// 128 threads), or with 128 threads holding two virtual threads each (V = 2)
// for long ones, where smaller CTAs keep more rows, and so more bytes, in
// flight per SM (15,860 rows: 75 -> 64 us, 67 -> 79 % of HBM).  Both give
// the same bits.
constexpr int MOD_VT = 256;                      // virtual threads per row
constexpr int MOD_MAXC = 4;                      // chunks per virtual thread: D <= 256 * 4 * 8 = 8192
constexpr int kModulateLongRows = 4096;
}  // namespace

template <int V>
__global__ void __launch_bounds__(MOD_VT / V) modulate_kernel(const ModulateArgs a) {
  constexpr int NT = MOD_VT / V;                 // real threads
  const int row = blockIdx.x;
  griddep_launch_dependents();
  griddep_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __shared__ float red[MOD_VT / 32];
  const int tg = a.tag[row], ti = a.tidx[row];
  if ((unsigned)tg > 2u || (unsigned)ti >= (unsigned)a.T) {
    if (threadIdx.x == 0) record_error(a.err, DEVERR_INDEX);
    return;
  }
  const int nch = a.D >> 3;
  const __nv_bfloat16* trow_chk = a.table + (size_t)(ti * 3 + tg) * 6 * a.D;
  if (!in_bounds<__nv_bfloat16>(a.x, a.x_elems, a.x + (size_t)row * a.D, a.D, a.err, 14) ||
      !in_bounds<__nv_bfloat16>(a.table, a.table_elems, trow_chk, (size_t)6 * a.D, a.err, 15) ||
      !in_bounds<__nv_bfloat16>(a.h, a.h_elems, a.h + (size_t)row * a.D, a.D, a.err, 16))
    return;
  const uint4* xr = reinterpret_cast<const uint4*>(a.x + (size_t)row * a.D);
  uint4 xv[V][MOD_MAXC];
  float ss[V];
#pragma unroll
  for (int v = 0; v < V; ++v) {
    ss[v] = 0.0f;
    const int vt = threadIdx.x + v * NT;
#pragma unroll
    for (int i = 0; i < MOD_MAXC; ++i) {
      const int c = vt + i * MOD_VT;
      if (c < nch) {
        xv[v][i] = xr[c];
        const uint32_t w[4] = {xv[v][i].x, xv[v][i].y, xv[v][i].z, xv[v][i].w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float lo = bf16_lo(w[e]), hi = bf16_hi(w[e]);
          ss[v] = __fmaf_rn(lo, lo, ss[v]);
          ss[v] = __fmaf_rn(hi, hi, ss[v]);
        }
      }
    }
  }
#pragma unroll
  for (int v = 0; v < V; ++v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss[v] += __shfl_xor_sync(0xffffffffu, ss[v], o);
    if (lane == 0) red[warp + v * (NT / 32)] = ss[v];
  }
  __syncthreads();
  float tot = 0.0f;
#pragma unroll
  for (int w = 0; w < MOD_VT / 32; ++w) tot += red[w];
  const float inv = 1.0f / sqrtf(tot / (float)a.D + a.eps);

  const __nv_bfloat16* trow = a.table + (size_t)(ti * 3 + tg) * 6 * a.D;
  const uint4* shp = reinterpret_cast<const uint4*>(trow + (size_t)a.chunk_shift * a.D);
  const uint4* scp = reinterpret_cast<const uint4*>(trow + (size_t)a.chunk_scale * a.D);
  const uint4* gp = reinterpret_cast<const uint4*>(a.gain);
  uint4* hp = reinterpret_cast<uint4*>(a.h + (size_t)row * a.D);
#pragma unroll
  for (int v = 0; v < V; ++v) {
#pragma unroll
    for (int i = 0; i < MOD_MAXC; ++i) {
      const int c = threadIdx.x + v * NT + i * MOD_VT;
      if (c < nch) {
        const uint4 gv = gp[c], shv = shp[c], scv = scp[c];
        const uint32_t xw[4] = {xv[v][i].x, xv[v][i].y, xv[v][i].z, xv[v][i].w};
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
}

cudaError_t launch_modulate(const ModulateArgs& a, cudaStream_t stream) {
  const bool long_doc = a.S >= kModulateLongRows;
  cudaError_t e = long_doc ? launch_kernel(modulate_kernel<2>, dim3(a.S), dim3(MOD_VT / 2), 0, stream, a)
                           : launch_kernel(modulate_kernel<1>, dim3(a.S), dim3(MOD_VT), 0, stream, a);
  if (e != cudaSuccess) return e;
  set_kernel_info("modulate_kernel rows=%d threads=%d vec=16B reduce=fixed-tree(256)", a.S,
                  long_doc ? MOD_VT / 2 : MOD_VT);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Persistent CTAs (one per SM); a unit is the q and k of one packed row for a
// block of up to 64 heads.  Warp 0 streams units through a ring of shared
// memory stages with two 3-D TMA loads each ([row][head][128] boxes of q and
// of k) and, while they fly, computes the row's 48 rotation angles (bands
// t, h, w x 16 frequencies, fp32(pos) * omega_f in fp32) into the stage.
// Warps 1..16 take whole heads of a stage: lanes 0-15 hold q, lanes 16-31
// hold k, lane l of a half owning channels 8l..8l+7.  The rotation pairs
// channel j < 48 with j + 48, i.e. half-lane l < 6 with l + 6 (one shuffle);
// half-lanes 12-15 carry the 32 pass-through channels.  Results go straight
// back to global memory (in place) with 16-byte stores.
constexpr int ROPE_CWARPS = 16;
constexpr int ROPE_THREADS = 32 * (ROPE_CWARPS + 1);
constexpr int ROPE_MAX_HB = 64;

__host__ __device__ inline int rope_heads_per_unit(int H) {
  const int nb = (H + ROPE_MAX_HB - 1) / ROPE_MAX_HB;
  return (H + nb - 1) / nb;
}
__host__ __device__ inline int rope_stage_bytes(int hb) { return 2 * hb * 256; }
__host__ __device__ inline int rope_stages(int hb) {
  const int st = (192 * 1024) / rope_stage_bytes(hb);
  return st > 8 ? 8 : st;
}
__host__ __device__ inline int rope_smem_bytes(int hb) {
  const int st = rope_stages(hb);
  return 128 + st * rope_stage_bytes(hb) + st * (96 * 4 + 16) + 2 * st * 8 + 16;
}

__global__ void __launch_bounds__(ROPE_THREADS, 1)
    rope_qknorm_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                       const RopeArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((128u - (smem_u32(smem_raw) & 127u)) & 127u);
  const int HB = rope_heads_per_unit(a.H);
  const int nhb = (a.H + HB - 1) / HB;
  const int STAGES = rope_stages(HB);
  const int SB = rope_stage_bytes(HB);
  uint8_t* tiles = smem;                                            // [STAGES][q|k][HB][128] bf16
  float* ang = reinterpret_cast<float*>(tiles + STAGES * SB);        // [STAGES][cos 48 | sin 48]
  int* bad = reinterpret_cast<int*>(ang + STAGES * 96);              // [STAGES]
  uint64_t* full = reinterpret_cast<uint64_t*>(
      reinterpret_cast<uint8_t*>(ang) + STAGES * (96 * 4 + 16));     // 8-byte aligned
  uint64_t* empty = full + STAGES;
  int* abort_flag = reinterpret_cast<int*>(empty + STAGES);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long units = (long long)a.S * nhb;

  griddep_launch_dependents();
  if (threadIdx.x == 0) {
    for (int st = 0; st < STAGES; ++st) {
      mbar_init(&full[st], 2);               // expect_tx arrival + angles-ready arrival
      mbar_init(&empty[st], ROPE_CWARPS);
    }
    *abort_flag = timeout_recorded(a.err) ? 1 : 0;   // sticky timeout of an earlier launch
    fence_mbar_init();
  }
  if (threadIdx.x == 32) {
    tma_prefetch_desc(&tmq);
    tma_prefetch_desc(&tmk);
  }
  __syncthreads();
  griddep_wait();
  const WaitCtl abort_v{abort_flag, a.err, KID_ROPE};

  // a wait of an earlier launch ran out (sticky until h3_sync_check; read
  // in the prologue, beside the previous kernel): this launch skips its
  // work, before any copy or MMA is issued
  const bool skip = *abort_v.flag != 0;

  if (skip) {
  } else if (warp == 0) {
    // ------------------------------------------------------------ producer
    int stage = 0;
    uint32_t phase = 0;
    int last_phase[8];
    for (int st = 0; st < 8; ++st) last_phase[st] = -1;
    bool ok = true;
    for (long long u = blockIdx.x; u < units; u += gridDim.x) {
      const int row = (int)(u / nhb), h0 = (int)(u % nhb) * HB;
      // every lane waits (and so acquires the stage); the outcome is made warp-uniform
      if (!__all_sync(0xffffffffu, mbar_wait(&empty[stage], phase ^ 1u, abort_v))) { ok = false; break; }
      if (lane == 0) {
        uint8_t* t = tiles + stage * SB;
        mbar_arrive_expect_tx(&full[stage], (uint32_t)SB);
        tma_load_3d(t, &tmq, &full[stage], 0, h0, row);
        tma_load_3d(t + SB / 2, &tmk, &full[stage], 0, h0, row);
        last_phase[stage] = (int)phase;
      }
      if (lane < 16) {
        int anybad = 0;
#pragma unroll
        for (int band = 0; band < 3; ++band) {
          const int p = a.pos[(size_t)row * 3 + band];
          anybad |= (unsigned)p >= (1u << 24);
          float sn, cs;
          sincosf((float)p * a.omega[lane], &sn, &cs);
          ang[stage * 96 + band * 16 + lane] = cs;
          ang[stage * 96 + 48 + band * 16 + lane] = sn;
        }
        anybad = __any_sync(0x0000ffffu, anybad);
        if (lane == 0) bad[stage] = anybad;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&full[stage]);
      if (++stage == STAGES) { stage = 0; phase ^= 1u; }
    }
    if (!ok && lane == 0) {   // let every load already issued land before the CTA exits
      const uint64_t t0 = globaltimer();
      for (int st = 0; st < STAGES; ++st) {
        if (last_phase[st] < 0) continue;
        while (!mbar_try_wait(&full[st], (uint32_t)last_phase[st]))
          if (globaltimer() - t0 > kWaitLimitNs) break;
      }
    }
  } else {
    // ------------------------------------------------------------ compute
    const int cw = warp - 1;
    const int hl = lane & 15;
    const bool is_k = lane >= 16;
    const int partner = hl < 6 ? lane + 6 : (hl < 12 ? lane - 6 : lane);
    const int col = hl < 12 ? (hl % 6) * 8 : 0;                 // first rotation column of the lane
    const float sgn = hl < 6 ? -1.0f : 1.0f;
    // channel pairs (2e, 2e+1) of the lane's 8 channels travel as float2 so
    // the per-channel products run as packed fp32 (IEEE, per lane)
    float2 g2[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const __nv_bfloat16* gp = (is_k ? a.k_gain : a.q_gain) + hl * 8 + 2 * e;
      g2[e] = make_float2(__bfloat162float(gp[0]), __bfloat162float(gp[1]));
    }
    __nv_bfloat16* gbase = is_k ? a.k : a.q;
    int stage = 0;
    uint32_t phase = 0;
    for (long long u = blockIdx.x; u < units; u += gridDim.x) {
      const int row = (int)(u / nhb), h0 = (int)(u % nhb) * HB;
      if (!__all_sync(0xffffffffu, mbar_wait(&full[stage], phase, abort_v))) break;
      if (bad[stage]) {
        if (cw == 0 && lane == 0) record_error(a.err, DEVERR_INDEX);
      } else {
        float2 cs2[4], sn2[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          if (hl < 12) {
            cs2[e] = make_float2(ang[stage * 96 + col + 2 * e], ang[stage * 96 + col + 2 * e + 1]);
            sn2[e] = make_float2(sgn * ang[stage * 96 + 48 + col + 2 * e], sgn * ang[stage * 96 + 48 + col + 2 * e + 1]);
          } else {
            cs2[e] = make_float2(1.0f, 1.0f);
            sn2[e] = make_float2(0.0f, 0.0f);
          }
        }
        const uint8_t* t = tiles + stage * SB + (is_k ? SB / 2 : 0) + hl * 16;
        // two heads per pass (h and h + ROPE_CWARPS), interleaved for ILP
        for (int h = cw; h < HB && h0 + h < a.H; h += 2 * ROPE_CWARPS) {
          const int hh[2] = {h, h + ROPE_CWARPS};
          const bool second = hh[1] < HB && h0 + hh[1] < a.H;   // warp-uniform
          float2 v[2][4];
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            uint4 r = make_uint4(0u, 0u, 0u, 0u);
            if (j == 0 || second) r = *reinterpret_cast<const uint4*>(t + hh[j] * 256);
            const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) v[j][e] = make_float2(bf16_lo(w[e]), bf16_hi(w[e]));
          }
          // sum of squares: even and odd channels in two lanes of a float2,
          // then added, then reduced over the 16 lanes of the half
          float ss[2];
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            float2 acc = make_float2(0.0f, 0.0f);
#pragma unroll
            for (int e = 0; e < 4; ++e) acc = __ffma2_rn(v[j][e], v[j][e], acc);
            ss[j] = acc.x + acc.y;
          }
#pragma unroll
          for (int o = 8; o > 0; o >>= 1)
#pragma unroll
            for (int j = 0; j < 2; ++j) ss[j] += __shfl_xor_sync(0xffffffffu, ss[j], o);   // within the half
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            const float inv = 1.0f / sqrtf(ss[j] * (1.0f / 128.0f) + a.eps);
            const float2 inv2 = make_float2(inv, inv);
            uint32_t nb[4], ob[4], outw[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {   // normed channels, rounded to bf16 (two per word)
              const float2 x = __fmul2_rn(__fmul2_rn(v[j][e], inv2), g2[e]);
              nb[e] = pack_bf16x2(x.x, x.y);
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) ob[e] = __shfl_sync(0xffffffffu, nb[e], partner);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 n = make_float2(bf16_lo(nb[e]), bf16_hi(nb[e]));
              const float2 other = make_float2(bf16_lo(ob[e]), bf16_hi(ob[e]));
              const float2 y = __ffma2_rn(n, cs2[e], __fmul2_rn(other, sn2[e]));
              outw[e] = pack_bf16x2(y.x, y.y);
            }
            __nv_bfloat16* gp = gbase + (size_t)row * a.row_stride + (size_t)(h0 + hh[j]) * a.head_stride + hl * 8;
            if ((j == 0 || second) && in_bounds<__nv_bfloat16>(gbase, a.qk_elems, gp, 8, a.err, 17))
              *reinterpret_cast<uint4*>(gp) = make_uint4(outw[0], outw[1], outw[2], outw[3]);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[stage]);
      if (++stage == STAGES) { stage = 0; phase ^= 1u; }
    }
  }
  __syncthreads();
  if (threadIdx.x == 0 && *abort_v.flag) record_error(a.err, DEVERR_TIMEOUT);
}

int rope_qknorm_smem_bytes(int H) { return rope_smem_bytes(rope_heads_per_unit(H)); }
int rope_qknorm_heads_per_unit(int H) { return rope_heads_per_unit(H); }

cudaError_t launch_rope_qknorm(const CUtensorMap& tmq, const CUtensorMap& tmk, const RopeArgs& a,
                               int num_sms, cudaStream_t stream) {
  const int hb = rope_heads_per_unit(a.H);
  const int smem = rope_smem_bytes(hb);
  cudaError_t e = cudaFuncSetAttribute(rope_qknorm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const long long units = (long long)a.S * ((a.H + hb - 1) / hb);
  const int grid = (int)(units < num_sms ? units : num_sms);
  e = launch_kernel(rope_qknorm_kernel, dim3(grid), dim3(ROPE_THREADS), smem, stream, tmq, tmk, a);
  if (e != cudaSuccess) return e;
  set_kernel_info("rope_qknorm_kernel persistent tma-3d units=%lld heads/unit=%d stages=%d grid=%d", units, hb,
                  rope_stages(hb), grid);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Token refiner set-up: the block's kernels run the refiner when the AdaLN
// table is the identity modulation (shift 0, scale 0, gate 1 in all six
// chunks of the three modality rows of timestep 0) and every row is a text
// row at timestep 0 and position (0, 0, 0), where MM-RoPE is the identity.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) refiner_setup_kernel(int S, int D, __nv_bfloat16* __restrict__ table,
                                                            int32_t* __restrict__ tag, int32_t* __restrict__ tidx,
                                                            int32_t* __restrict__ pos, uint32_t* zero_words,
                                                            int n_zero) {
  griddep_launch_dependents();
  griddep_wait();
  // the stream-K flags of the call
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n_zero; i += gridDim.x * blockDim.x) zero_words[i] = 0u;
  const int n_tab = 3 * 6 * D;
  const int n = n_tab + 5 * S;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
    if (i < n_tab) {
      const int chunk = (i / D) % 6;
      table[i] = __float2bfloat16_rn((chunk == 2 || chunk == 5) ? 1.0f : 0.0f);
    } else {
      const int j = i - n_tab;
      if (j < S) tag[j] = 1;             // text
      else if (j < 2 * S) tidx[j - S] = 0;
      else pos[j - 2 * S] = 0;
    }
  }
}

cudaError_t launch_refiner_setup(int S, int D, __nv_bfloat16* table, int32_t* tag, int32_t* tidx, int32_t* pos,
                                 uint32_t* zero_words, int n_zero_words, cudaStream_t st) {
  const long long n = 18LL * D + 5LL * S;
  int grid = (int)((n + 255) / 256);
  if (grid > 4 * num_sms()) grid = 4 * num_sms();
  cudaError_t e = launch_kernel(refiner_setup_kernel, dim3(grid), dim3(256), 0, st, S, D, table, tag, tidx, pos,
                                zero_words, zero_words ? n_zero_words : 0);
  if (e != cudaSuccess) return e;
  set_kernel_info("refiner_setup_kernel identity-table rows=%d", S);
  return cudaGetLastError();
}

}  // namespace h3
