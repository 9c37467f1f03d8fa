// tcgen05 GEMMs for the H3 block projections.
//
// gemm_bf16_tc<EPI>: D[128 x 256] tiles of  act[M][K] . W[rows][K]^T, bf16 in,
// fp32 accumulate in TMEM, with the epilogue fused per projection:
//   EPI_PLAIN   y = bf16(acc + b)
//   EPI_QKV     q|k tiles of one head: per-head Q/K RMSNorm, then the partial
//               three-axis MM-RoPE on 96 of the 128 channels (RFC section 4:
//               norm before RoPE); v tiles plain
//   EPI_RESID   y = bf16(x + gate[r] * bf16(acc + b))   (RFC s4 residual order)
//   EPI_SWIGLU  a = bf16(SiLU(g) * u) with g, u the paired gate / value tiles
//               (the h3-metal README, section "Metal 4 and TensorOps paths",
//               pairs the FC1 gate and up tiles so SwiGLU happens before the
//               store)
// Structure: persistent CTAs (one per SM), static tile order (m fastest so CTAs
// running together share the weight tile through L2), warp 0 issues TMA loads
// into a 4-stage mbarrier ring, warp 1 issues tcgen05.mma from one thread into
// one of two TMEM accumulators (2 x 256 columns), warps 2-5 drain the other
// accumulator through tcgen05.ld and run the epilogue.  The K loop of a tile
// is a fixed sequence of 16-deep MMAs: no split-K, so the reduction order is
// independent of M and of the grid.
//
// adaln_table_kernel: the AdaLN projection.  Its M dimension is only T <= 16
// timestep rows, so the GEMM is run transposed: the 18*D weight rows are the
// 128-row M operand streamed by TMA, and bf16(SiLU(t_cond)) -- computed by the
// CTA itself into shared memory -- is the resident N = 16 operand.  The
// kernel is bound by the weight stream from HBM.
#include "h3_device.cuh"
#include "h3_internal.h"

#include <cstdio>

namespace h3 {

namespace {

constexpr int BM = 128, BN = 256, BK = 64, STAGES = 4;
constexpr int A_STAGE_BYTES = BM * BK * 2;   // 16 KB
constexpr int B_STAGE_BYTES = BN * BK * 2;   // 32 KB
constexpr int GEMM_THREADS = 192;
constexpr int GEMM_SMEM = 1024 + STAGES * (A_STAGE_BYTES + B_STAGE_BYTES) + 256;

struct GemmSmem {
  uint8_t* a;
  uint8_t* b;
  uint64_t* full;
  uint64_t* empty;
  uint64_t* acc_full;
  uint64_t* acc_empty;
  uint64_t* drain;
  uint32_t* tmem_slot;
  int* abort_flag;
};

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  const uint32_t s = smem_u32(p);
  return p + (((s + 1023u) & ~1023u) - s);
}

// Bounded wait that ignores the abort flag (used to drain in-flight work).
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer() - t0 > kWaitLimitNs) return;
  }
}

__device__ __forceinline__ void tmem_ld_wait16(uint32_t (&r)[16]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),
                 "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]),
                 "+r"(r[14]), "+r"(r[15])::"memory");
}

__device__ __forceinline__ float bias_at(const __nv_bfloat16* b, int i) {
  return b ? __bfloat162float(b[i]) : 0.0f;
}

// Weight rows of the two 128-row halves of the B tile n_blk.
template <int EPI>
__device__ __forceinline__ void b_rows(const GemmArgs& a, int n_blk, int& r0, int& r1) {
  if (EPI == EPI_SWIGLU) {
    r0 = n_blk * 128;            // gate rows
    r1 = a.F + n_blk * 128;      // value rows
  } else if (EPI == EPI_QKV) {
    if (n_blk < a.H) {           // q | k of head n_blk
      r0 = n_blk * 384;
      r1 = r0 + 128;
    } else {                     // v of heads 2p, 2p+1
      const int p = n_blk - a.H;
      r0 = (2 * p) * 384 + 256;
      r1 = (2 * p + 1) * 384 + 256;
    }
  } else {
    r0 = n_blk * 256;
    r1 = r0 + 128;
  }
}

// ---------------------------------------------------------------------------
// epilogues (4 warps, thread = one accumulator row)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void store32_bf16(__nv_bfloat16* dst, const float (&v)[32]) {
  uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    uint4 w;
    w.x = pack_bf16x2(v[g * 8 + 0], v[g * 8 + 1]);
    w.y = pack_bf16x2(v[g * 8 + 2], v[g * 8 + 3]);
    w.z = pack_bf16x2(v[g * 8 + 4], v[g * 8 + 5]);
    w.w = pack_bf16x2(v[g * 8 + 6], v[g * 8 + 7]);
    d[g] = w;
  }
}
__device__ __forceinline__ void store16_bf16(__nv_bfloat16* dst, const float (&v)[16]) {
  uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int g = 0; g < 2; ++g) {
    uint4 w;
    w.x = pack_bf16x2(v[g * 8 + 0], v[g * 8 + 1]);
    w.y = pack_bf16x2(v[g * 8 + 2], v[g * 8 + 3]);
    w.z = pack_bf16x2(v[g * 8 + 4], v[g * 8 + 5]);
    w.w = pack_bf16x2(v[g * 8 + 6], v[g * 8 + 7]);
    d[g] = w;
  }
}

__device__ __forceinline__ void epi_plain(const GemmArgs& a, uint32_t tacc, int m, bool valid, int n_blk) {
#pragma unroll 1
  for (int c = 0; c < BN / 32; ++c) {
    uint32_t r[32];
    tmem_ld32(tacc + c * 32, r);
    tmem_ld_wait(r);
    const int n0 = n_blk * BN + c * 32;
    if (valid) {
      __nv_bfloat16* dst = a.out + (size_t)m * a.ldo + n0;
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        const int n = n0 + g * 8;
        if (n < a.n_valid) {
          uint4 w;
          uint32_t* wp = reinterpret_cast<uint32_t*>(&w);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float lo = __uint_as_float(r[g * 8 + 2 * e]) + bias_at(a.bias, n + 2 * e);
            const float hi = __uint_as_float(r[g * 8 + 2 * e + 1]) + bias_at(a.bias, n + 2 * e + 1);
            wp[e] = pack_bf16x2(lo, hi);
          }
          *reinterpret_cast<uint4*>(dst + g * 8) = w;
        }
      }
    }
  }
}

__device__ __forceinline__ void epi_resid(const GemmArgs& a, uint32_t tacc, int m, bool valid, int n_blk) {
  const __nv_bfloat16* gate = nullptr;
  if (valid) {
    const int tg = a.tag[m], ti = a.tidx[m];
    if ((unsigned)tg > 2u || (unsigned)ti >= (unsigned)a.T) {
      record_error(a.err, DEVERR_INDEX);
      valid = false;
    } else {
      gate = a.table + ((size_t)(ti * 3 + tg) * 6 + a.chunk) * a.D;
    }
  }
#pragma unroll 1
  for (int c = 0; c < BN / 32; ++c) {
    uint32_t r[32];
    tmem_ld32(tacc + c * 32, r);
    tmem_ld_wait(r);
    const int n0 = n_blk * BN + c * 32;
    if (valid && n0 < a.n_valid) {
      const uint4* xs = reinterpret_cast<const uint4*>(a.resid + (size_t)m * a.ldr + n0);
      const uint4* gs = reinterpret_cast<const uint4*>(gate + n0);
      uint4* dst = reinterpret_cast<uint4*>(a.out + (size_t)m * a.ldo + n0);
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        const uint4 xv = xs[g], gv = gs[g];
        const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
        const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w};
        uint32_t ow[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int j = g * 8 + 2 * e;
          const float flo = bf16_round(__uint_as_float(r[j]) + bias_at(a.bias, n0 + j));
          const float fhi = bf16_round(__uint_as_float(r[j + 1]) + bias_at(a.bias, n0 + j + 1));
          const float ylo = __fmaf_rn(bf16_lo(gw[e]), flo, bf16_lo(xw[e]));
          const float yhi = __fmaf_rn(bf16_hi(gw[e]), fhi, bf16_hi(xw[e]));
          ow[e] = pack_bf16x2(ylo, yhi);
        }
        dst[g] = make_uint4(ow[0], ow[1], ow[2], ow[3]);
      }
    }
  }
}

__device__ __forceinline__ void epi_swiglu(const GemmArgs& a, uint32_t tacc, int m, bool valid, int n_blk) {
#pragma unroll 1
  for (int c = 0; c < 4; ++c) {
    uint32_t g[32], u[32];
    tmem_ld32(tacc + c * 32, g);
    tmem_ld32(tacc + 128 + c * 32, u);
    tmem_ld_wait(g);
    tmem_ld_wait(u);
    const int n0 = n_blk * 128 + c * 32;
    if (valid) {
      float v[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const float gv = bf16_round(__uint_as_float(g[j]) + bias_at(a.bias, n0 + j));
        const float uv = bf16_round(__uint_as_float(u[j]) + bias_at(a.bias, a.F + n0 + j));
        v[j] = (gv / (1.0f + expf(-gv))) * uv;
      }
      store32_bf16(a.out + (size_t)m * a.ldo + n0, v);
    }
  }
}

// q|k tile of head h: columns [0,128) q, [128,256) k.
__device__ __forceinline__ void epi_qk(const GemmArgs& a, uint32_t tacc, int m, bool valid, int h) {
  float pos[3] = {0.f, 0.f, 0.f};
  if (valid) {
#pragma unroll
    for (int ax = 0; ax < 3; ++ax) {
      const int p = a.pos[(size_t)m * 3 + ax];
      if ((unsigned)p >= (1u << 24)) {
        record_error(a.err, DEVERR_INDEX);
        valid = false;
      }
      pos[ax] = (float)p;
    }
  }
  const int colq = h * 384;  // output column of q; k at +128
  // pass 1: per-head sums of squares of the bf16-cast projections
  float ss[2] = {0.f, 0.f};
#pragma unroll 1
  for (int part = 0; part < 2; ++part) {
#pragma unroll 1
    for (int c = 0; c < 4; ++c) {
      uint32_t r[32];
      tmem_ld32(tacc + part * 128 + c * 32, r);
      tmem_ld_wait(r);
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const float v = bf16_round(__uint_as_float(r[j]) + bias_at(a.bias, colq + part * 128 + c * 32 + j));
        ss[part] = __fmaf_rn(v, v, ss[part]);
      }
    }
  }
  float inv[2];
  inv[0] = 1.0f / sqrtf(ss[0] * (1.0f / 128.0f) + a.eps);
  inv[1] = 1.0f / sqrtf(ss[1] * (1.0f / 128.0f) + a.eps);
  // pass 2: normalise, rotate the 96 rotary channels, pass 32 through
#pragma unroll 1
  for (int band = 0; band < 3; ++band) {
    float cs[16], sn[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float ang = pos[band] * a.omega[i];
      sincosf(ang, &sn[i], &cs[i]);
    }
#pragma unroll 1
    for (int part = 0; part < 2; ++part) {
      const __nv_bfloat16* gain = part ? a.k_gain : a.q_gain;
      uint32_t lo[16], hi[16];
      tmem_ld16(tacc + part * 128 + band * 16, lo);
      tmem_ld16(tacc + part * 128 + 48 + band * 16, hi);
      tmem_ld_wait(lo, hi);
      if (valid) {
        float o1[16], o2[16];
        const int cb = colq + part * 128;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int j = band * 16 + i;
          const float v1 = bf16_round(__uint_as_float(lo[i]) + bias_at(a.bias, cb + j));
          const float v2 = bf16_round(__uint_as_float(hi[i]) + bias_at(a.bias, cb + 48 + j));
          const float x1 = bf16_round(v1 * inv[part] * __bfloat162float(gain[j]));
          const float x2 = bf16_round(v2 * inv[part] * __bfloat162float(gain[48 + j]));
          o1[i] = __fmaf_rn(x1, cs[i], -(x2 * sn[i]));
          o2[i] = __fmaf_rn(x2, cs[i], x1 * sn[i]);
        }
        __nv_bfloat16* dst = a.out + (size_t)m * a.ldo + cb;
        store16_bf16(dst + band * 16, o1);
        store16_bf16(dst + 48 + band * 16, o2);
      }
    }
  }
#pragma unroll 1
  for (int part = 0; part < 2; ++part) {
    const __nv_bfloat16* gain = part ? a.k_gain : a.q_gain;
    uint32_t r[32];
    tmem_ld32(tacc + part * 128 + 96, r);
    tmem_ld_wait(r);
    if (valid) {
      const int cb = colq + part * 128;
      float v[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const float x = bf16_round(__uint_as_float(r[j]) + bias_at(a.bias, cb + 96 + j));
        v[j] = x * inv[part] * __bfloat162float(gain[96 + j]);
      }
      store32_bf16(a.out + (size_t)m * a.ldo + cb + 96, v);
    }
  }
}

// v tile: columns [0,128) v of head 2p, [128,256) v of head 2p+1.
__device__ __forceinline__ void epi_v(const GemmArgs& a, uint32_t tacc, int m, bool valid, int p) {
#pragma unroll 1
  for (int half = 0; half < 2; ++half) {
    const int head = 2 * p + half;
#pragma unroll 1
    for (int c = 0; c < 4; ++c) {
      uint32_t r[32];
      tmem_ld32(tacc + half * 128 + c * 32, r);
      tmem_ld_wait(r);
      if (valid && head < a.H) {
        const int cb = head * 384 + 256 + c * 32;
        float v[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]) + bias_at(a.bias, cb + j);
        store32_bf16(a.out + (size_t)m * a.ldo + cb, v);
      }
    }
  }
}

template <int EPI>
__device__ __forceinline__ void run_epilogue(const GemmArgs& a, uint32_t tacc, int m_blk, int n_blk, int row) {
  const int m = m_blk * BM + row;
  const bool valid = m < a.M;
  if (EPI == EPI_PLAIN) epi_plain(a, tacc, m, valid, n_blk);
  if (EPI == EPI_RESID) epi_resid(a, tacc, m, valid, n_blk);
  if (EPI == EPI_SWIGLU) epi_swiglu(a, tacc, m, valid, n_blk);
  if (EPI == EPI_QKV) {
    if (n_blk < a.H) epi_qk(a, tacc, m, valid, n_blk);
    else epi_v(a, tacc, m, valid, n_blk - a.H);
  }
}

}  // namespace

template <int EPI>
__global__ void __launch_bounds__(GEMM_THREADS, 1)
    gemm_bf16_tc(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                 const GemmArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * A_STAGE_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sB + STAGES * B_STAGE_BYTES);
  uint64_t* full = bars;
  uint64_t* empty = bars + STAGES;
  uint64_t* acc_full = bars + 2 * STAGES;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* drain = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], 4);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) tmem_alloc(tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int num_tiles = args.num_m * args.num_n;
  volatile int* abort_v = abort_flag;

  if (warp == 0) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int last_phase[STAGES];
      for (int s = 0; s < STAGES; ++s) last_phase[s] = -1;
      bool ok = true;
      for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
        const int m_blk = tile % args.num_m, n_blk = tile / args.num_m;
        int r0, r1;
        b_rows<EPI>(args, n_blk, r0, r1);
        for (int kb = 0; kb < args.num_k; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, abort_v)) { ok = false; break; }
          mbar_arrive_expect_tx(&full[stage], A_STAGE_BYTES + B_STAGE_BYTES);
          uint8_t* b = sB + stage * B_STAGE_BYTES;
          tma_load_2d(sA + stage * A_STAGE_BYTES, &tmA, &full[stage], kb * BK, m_blk * BM);
          tma_load_2d(b, &tmB, &full[stage], kb * BK, r0);
          tma_load_2d(b + B_STAGE_BYTES / 2, &tmB, &full[stage], kb * BK, r1);
          last_phase[stage] = (int)phase;
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
      }
      if (!ok) {  // let every load already issued land before the CTA exits
        for (int s = 0; s < STAGES; ++s)
          if (last_phase[s] >= 0) drain_wait(&full[s], (uint32_t)last_phase[s]);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16(BM, BN);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      int it = 0;
      for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x, ++it) {
        const int acc = it & 1;
        const uint32_t acc_phase = (uint32_t)(it >> 1) & 1u;
        if (!mbar_wait(&acc_empty[acc], acc_phase ^ 1u, abort_v)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
        for (int kb = 0; kb < args.num_k; ++kb) {
          if (!mbar_wait(&full[stage], phase, abort_v)) { ok = false; break; }
          tc_fence_after();
          const uint32_t a0 = smem_u32(sA + stage * A_STAGE_BYTES);
          const uint32_t b0 = smem_u32(sB + stage * B_STAGE_BYTES);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k) {
            mma_bf16_ss(d_tmem, sdesc_kmajor(a0 + k * 32), sdesc_kmajor(b0 + k * 32), idesc,
                        (kb | k) != 0 ? 1u : 0u);
          }
          mma_commit(&empty[stage]);
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        mma_commit(&acc_full[acc]);
      }
      if (!ok) {  // all MMAs issued so far must finish before TMEM is released
        mma_commit(drain);
        drain_wait(drain, 0);
      }
    }
    __syncwarp();
  } else {
    const int q = warp & 3;
    const int row = q * 32 + lane;
    int it = 0;
    for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x, ++it) {
      const int acc = it & 1;
      const uint32_t acc_phase = (uint32_t)(it >> 1) & 1u;
      if (!mbar_wait(&acc_full[acc], acc_phase, abort_v)) break;
      tc_fence_after();
      const int m_blk = tile % args.num_m, n_blk = tile / args.num_m;
      const uint32_t tacc = tmem_addr(tmem_base, (uint32_t)(q * 32), (uint32_t)(acc * BN));
      run_epilogue<EPI>(args, tacc, m_blk, n_blk, row);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[acc]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0 && *abort_v) record_error(args.err, DEVERR_TIMEOUT);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 512);
  }
}

cudaError_t launch_gemm(int epi, const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmArgs& a,
                        cudaStream_t stream) {
  const int tiles = a.num_m * a.num_n;
  const int grid = tiles < num_sms() ? tiles : num_sms();
  const char* names[4] = {"plain", "qkv_qknorm_rope", "gated_residual", "swiglu"};
  cudaError_t e = cudaSuccess;
#define H3_LAUNCH_GEMM(E)                                                                          \
  case E: {                                                                                        \
    e = cudaFuncSetAttribute(gemm_bf16_tc<E>, cudaFuncAttributeMaxDynamicSharedMemorySize, GEMM_SMEM); \
    if (e != cudaSuccess) return e;                                                                \
    gemm_bf16_tc<E><<<grid, GEMM_THREADS, GEMM_SMEM, stream>>>(tmA, tmB, a);                       \
    break;                                                                                         \
  }
  switch (epi) {
    H3_LAUNCH_GEMM(EPI_PLAIN)
    H3_LAUNCH_GEMM(EPI_QKV)
    H3_LAUNCH_GEMM(EPI_RESID)
    H3_LAUNCH_GEMM(EPI_SWIGLU)
    default:
      return cudaErrorInvalidValue;
  }
#undef H3_LAUNCH_GEMM
  set_kernel_info("gemm_bf16_tc<%s> tcgen05.mma.cta_group::1.kind::f16 tile=%dx%dx%d stages=%d acc=f32 "
                  "tmem=2x%d grid=%d tiles=%dx%d k_blocks=%d",
                  names[epi], BM, BN, BK, STAGES, BN, grid, a.num_m, a.num_n, a.num_k);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// AdaLN table
// ---------------------------------------------------------------------------
namespace {
constexpr int AD_STAGES = 8;
constexpr int AD_BN = 16;
constexpr int AD_THREADS = 192;
constexpr int AD_U_MAX_KB = 44;  // cond_dim <= 44 * 64 = 2816
constexpr int AD_SMEM = 1024 + AD_U_MAX_KB * 2048 + AD_STAGES * A_STAGE_BYTES + 256;
}  // namespace

__global__ void __launch_bounds__(AD_THREADS, 1)
    adaln_table_kernel(const __grid_constant__ CUtensorMap tmW, const AdalnArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  const int nkb = args.C / BK;
  uint8_t* sU = smem;                         // nkb blocks of 16 rows x 128 B
  uint8_t* sA = smem + nkb * 2048;            // 1024-aligned (2048 multiple)
  uint64_t* bars = reinterpret_cast<uint64_t*>(sA + AD_STAGES * A_STAGE_BYTES);
  uint64_t* full = bars;
  uint64_t* empty = bars + AD_STAGES;
  uint64_t* acc_full = bars + 2 * AD_STAGES;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* drain = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < AD_STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], 4);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) tma_prefetch_desc(&tmW);
  if (warp == 1) tmem_alloc(tmem_slot, 32);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int num_tiles = args.NW / BM;
  volatile int* abort_v = abort_flag;
  if (warp != 0) {
    // Warps 1-5: u = bf16(SiLU(t_cond)) in fp32, rows >= T zero, written in
    // the K-major 128-byte-swizzled layout the tensor core reads, while warp 0
    // already streams weight tiles.
    for (int idx = threadIdx.x - 32; idx < AD_BN * args.C; idx += AD_THREADS - 32) {
      const int t = idx / args.C, k = idx - t * args.C;
      float v = 0.0f;
      if (t < args.T) {
        const float x = args.t_cond[(size_t)t * args.C + k];
        v = x / (1.0f + expf(-x));
      }
      const uint32_t off = (uint32_t)(k >> 6) * 2048u +
                           sw128_offset((uint32_t)t, (uint32_t)((k & 63) >> 3)) + (uint32_t)(k & 7) * 2u;
      *reinterpret_cast<__nv_bfloat16*>(sU + off) = __float2bfloat16_rn(v);
    }
    fence_proxy_async_smem();
    asm volatile("bar.sync 1, %0;" ::"n"(AD_THREADS - 32) : "memory");
  }

  if (warp == 0) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int last_phase[AD_STAGES];
      for (int s = 0; s < AD_STAGES; ++s) last_phase[s] = -1;
      bool ok = true;
      for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, abort_v)) { ok = false; break; }
          mbar_arrive_expect_tx(&full[stage], A_STAGE_BYTES);
          tma_load_2d(sA + stage * A_STAGE_BYTES, &tmW, &full[stage], kb * BK, tile * BM);
          last_phase[stage] = (int)phase;
          if (++stage == AD_STAGES) { stage = 0; phase ^= 1u; }
        }
      }
      if (!ok) {
        for (int s = 0; s < AD_STAGES; ++s)
          if (last_phase[s] >= 0) drain_wait(&full[s], (uint32_t)last_phase[s]);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16(BM, AD_BN);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      int it = 0;
      const uint32_t u0 = smem_u32(sU);
      for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x, ++it) {
        const int acc = it & 1;
        const uint32_t acc_phase = (uint32_t)(it >> 1) & 1u;
        if (!mbar_wait(&acc_empty[acc], acc_phase ^ 1u, abort_v)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * AD_BN);
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait(&full[stage], phase, abort_v)) { ok = false; break; }
          tc_fence_after();
          const uint32_t a0 = smem_u32(sA + stage * A_STAGE_BYTES);
          const uint32_t b0 = u0 + (uint32_t)kb * 2048u;
#pragma unroll
          for (int k = 0; k < BK / 16; ++k) {
            mma_bf16_ss(d_tmem, sdesc_kmajor(a0 + k * 32), sdesc_kmajor(b0 + k * 32), idesc,
                        (kb | k) != 0 ? 1u : 0u);
          }
          mma_commit(&empty[stage]);
          if (++stage == AD_STAGES) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        mma_commit(&acc_full[acc]);
      }
      if (!ok) {
        mma_commit(drain);
        drain_wait(drain, 0);
      }
    }
    __syncwarp();
  } else {
    const int q = warp & 3;
    const int row = q * 32 + lane;
    int it = 0;
    for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x, ++it) {
      const int acc = it & 1;
      const uint32_t acc_phase = (uint32_t)(it >> 1) & 1u;
      if (!mbar_wait(&acc_full[acc], acc_phase, abort_v)) break;
      tc_fence_after();
      uint32_t r[16];
      tmem_ld16(tmem_addr(tmem_base, (uint32_t)(q * 32), (uint32_t)(acc * AD_BN)), r);
      tmem_ld_wait16(r);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[acc]);
      const int n = tile * BM + row;
      const float b = bias_at(args.bias, n);
#pragma unroll
      for (int t = 0; t < AD_BN; ++t) {
        if (t < args.T) args.out[(size_t)t * args.NW + n] = __float2bfloat16_rn(__uint_as_float(r[t]) + b);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0 && *abort_v) record_error(args.err, DEVERR_TIMEOUT);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 32);
  }
}

cudaError_t launch_adaln_table(const CUtensorMap& tmW, const AdalnArgs& a, cudaStream_t stream) {
  const int tiles = a.NW / BM;
  const int grid = tiles < num_sms() ? tiles : num_sms();
  cudaError_t e = cudaFuncSetAttribute(adaln_table_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, AD_SMEM);
  if (e != cudaSuccess) return e;
  adaln_table_kernel<<<grid, AD_THREADS, AD_SMEM, stream>>>(tmW, a);
  set_kernel_info("adaln_table_kernel tcgen05.mma.cta_group::1.kind::f16 tile=%dx%dx%d stages=%d acc=f32 "
                  "tmem=2x%d grid=%d tiles=%d k_blocks=%d (SiLU prologue in smem)",
                  BM, AD_BN, BK, AD_STAGES, AD_BN, grid, tiles, a.C / BK);
  return cudaGetLastError();
}

}  // namespace h3
