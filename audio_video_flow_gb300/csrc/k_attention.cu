// Full non-causal attention over one packed document (RFC section 4: every row
// attends to every row, no mask), 128-wide heads, fp32 online softmax, on the
// 5th-generation tensor cores.
//
// One CTA computes one 128-row query tile of one head:
//   warp 0      TMA producer: Q once, then K_j and V_j tiles (128 rows x 128
//               channels, two 64-channel 128-byte-swizzled boxes each) into
//               rings of 3 (K) and 2 (V) tiles;
//   warp 1      MMA issuer (one thread): S_j = Q K_j^T into one of two TMEM
//               score buffers, and O += P_j V_j into the TMEM output
//               accumulator (V is read MN-major straight from its TMA tile);
//   warps 4-7   softmax, one query row per thread: tcgen05.ld of the score
//               row, running max and sum in fp32 (base-2 exponent with the
//               1/sqrt(128) scale folded in), P_j as bf16 into shared memory
//               in the tensor core's K-major layout, and the O rescale in TMEM
//               when the running max grows.
// S_{j+1} is computed while the softmax of tile j runs.  Keys past the end of
// the sequence (zero-filled by TMA) get probability 0; query rows past the end
// are computed and not stored.  Every sum runs in a fixed order, so the result
// does not depend on the grid or on other rows.
#include "h3_device.cuh"
#include "h3_internal.h"

#include <cmath>
#include <cstdlib>

namespace h3 {

namespace {
constexpr int AT_THREADS = 256;
constexpr int KV_TILE = 128;
constexpr int KST = 3, VST = 2;   // K ring 3 deep: K_{j+1} is loaded two steps ahead of its MMA
constexpr int TILE_BYTES = 128 * 128 * 2;   // 32 KB: two 16 KB boxes
constexpr int BOX_BYTES = 128 * 64 * 2;     // 16 KB
constexpr int AT_SMEM = 1024 + TILE_BYTES * (1 + KST + VST + 1) + 512;

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  const uint32_t s = smem_u32(p);
  return p + (((s + 1023u) & ~1023u) - s);
}
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer() - t0 > kWaitLimitNs) return;
  }
}
}  // namespace

__global__ void __launch_bounds__(AT_THREADS, 1)
    attention_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV, const AttnArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint8_t* sQ = smem;
  uint8_t* sK = sQ + TILE_BYTES;
  uint8_t* sV = sK + KST * TILE_BYTES;
  uint8_t* sP = sV + VST * TILE_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sP + TILE_BYTES);
  uint64_t* q_full = bars;
  uint64_t* k_full = bars + 1;
  uint64_t* k_empty = k_full + KST;
  uint64_t* v_full = k_empty + KST;
  uint64_t* v_empty = v_full + VST;
  uint64_t* s_full = v_empty + VST;
  uint64_t* s_empty = s_full + 2;
  uint64_t* p_full = s_empty + 2;
  uint64_t* o_done = p_full + 1;
  uint64_t* drain = o_done + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);

  griddep_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int q_tile = blockIdx.x, head = blockIdx.y;
  const int S = args.S;
  const int n_kv = (S + KV_TILE - 1) / KV_TILE;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < KST; ++s) { mbar_init(&k_full[s], 1); mbar_init(&k_empty[s], 1); }
    for (int s = 0; s < VST; ++s) { mbar_init(&v_full[s], 1); mbar_init(&v_empty[s], 1); }
    for (int b = 0; b < 2; ++b) { mbar_init(&s_full[b], 1); mbar_init(&s_empty[b], 4); }
    mbar_init(p_full, 4);
    mbar_init(o_done, 1);
    mbar_init(drain, 1);
    *abort_flag = timeout_recorded(args.err) ? 1 : 0;   // sticky timeout of an earlier launch
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  if (warp == 1) tmem_alloc(tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  griddep_wait();
  const uint32_t tmem_base = *tmem_slot;   // S0: cols [0,128), S1: [128,256), O: [256,384)
  const WaitCtl abort_v{abort_flag, args.err, KID_ATTN_1Q};

  // a wait of an earlier launch ran out (sticky until h3_sync_check; read
  // in the prologue, beside the previous kernel): this launch skips its
  // work, before any copy or MMA is issued
  const bool skip = *abort_v.flag != 0;

  if (skip) {
  } else if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      bool ok = true;
      int issued_k = 0, issued_v = 0;
      mbar_arrive_expect_tx(q_full, TILE_BYTES);
      tma_load_3d(sQ, &tmQ, q_full, 0, head, q_tile * 128);
      tma_load_3d(sQ + BOX_BYTES, &tmQ, q_full, 64, head, q_tile * 128);
      for (int j = 0; j < n_kv && ok; ++j) {
        const int ks = j % KST;
        const uint32_t kph = (uint32_t)(j / KST) & 1u;
        if (!mbar_wait(&k_empty[ks], kph ^ 1u, abort_v)) { ok = false; break; }
        mbar_arrive_expect_tx(&k_full[ks], TILE_BYTES);
        tma_load_3d(sK + ks * TILE_BYTES, &tmK, &k_full[ks], 0, head, j * KV_TILE);
        tma_load_3d(sK + ks * TILE_BYTES + BOX_BYTES, &tmK, &k_full[ks], 64, head, j * KV_TILE);
        ++issued_k;
        const int vs = j % VST;
        const uint32_t vph = (uint32_t)(j / VST) & 1u;
        if (!mbar_wait(&v_empty[vs], vph ^ 1u, abort_v)) { ok = false; break; }
        mbar_arrive_expect_tx(&v_full[vs], TILE_BYTES);
        tma_load_3d(sV + vs * TILE_BYTES, &tmV, &v_full[vs], 0, head, j * KV_TILE);
        tma_load_3d(sV + vs * TILE_BYTES + BOX_BYTES, &tmV, &v_full[vs], 64, head, j * KV_TILE);
        ++issued_v;
      }
      if (!ok) {  // let issued loads land before the CTA exits
        drain_wait(q_full, 0);
        for (int j = (issued_k > KST ? issued_k - KST : 0); j < issued_k; ++j)
          drain_wait(&k_full[j % KST], (uint32_t)(j / KST) & 1u);
        for (int j = (issued_v > VST ? issued_v - VST : 0); j < issued_v; ++j)
          drain_wait(&v_full[j % VST], (uint32_t)(j / VST) & 1u);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16(128, 128, false, false);
      constexpr uint32_t idesc_o = idesc_bf16(128, 128, false, true);   // V is MN-major
      const uint32_t q0 = smem_u32(sQ), k0 = smem_u32(sK), v0 = smem_u32(sV), p0 = smem_u32(sP);
      const uint32_t o_tmem = tmem_base + 256u;
      bool ok = mbar_wait(q_full, 0, abort_v);
      auto issue_s = [&](int j) -> bool {
        const int ks = j % KST;
        if (!mbar_wait(&k_full[ks], (uint32_t)(j / KST) & 1u, abort_v)) return false;
        const int b = j & 1;
        if (!mbar_wait(&s_empty[b], ((uint32_t)(j >> 1) & 1u) ^ 1u, abort_v)) return false;
        tc_fence_after();
        const uint32_t kb = k0 + (uint32_t)(ks * TILE_BYTES);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint32_t off = (uint32_t)((k >> 2) * BOX_BYTES + (k & 3) * 32);
          mma_bf16_ss(tmem_base + (uint32_t)(b * 128), sdesc_kmajor(q0 + off), sdesc_kmajor(kb + off), idesc_s,
                      k != 0 ? 1u : 0u);
        }
        mma_commit(&s_full[b]);
        mma_commit(&k_empty[ks]);
        return true;
      };
      if (ok) ok = issue_s(0);
      for (int j = 0; j < n_kv && ok; ++j) {
        if (j + 1 < n_kv && !issue_s(j + 1)) { ok = false; break; }
        if (!mbar_wait(p_full, (uint32_t)j & 1u, abort_v)) { ok = false; break; }
        const int vs = j % VST;
        if (!mbar_wait(&v_full[vs], (uint32_t)(j / VST) & 1u, abort_v)) { ok = false; break; }
        tc_fence_after();
        const uint32_t vb = v0 + (uint32_t)(vs * TILE_BYTES);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint64_t a_desc = sdesc_kmajor(p0 + (uint32_t)((k >> 2) * BOX_BYTES + (k & 3) * 32));
          // V tile: 128 key rows x 128 B per 64-channel box; 16 keys = 2048 B;
          // next 64 channels one box (16 KB) further: LBO = 16 KB, SBO = 1 KB.
          const uint64_t b_desc = sdesc_sw128(vb + (uint32_t)(k * 2048), BOX_BYTES, 1024);
          mma_bf16_ss(o_tmem, a_desc, b_desc, idesc_o, (j | k) != 0 ? 1u : 0u);
        }
        mma_commit(o_done);
        mma_commit(&v_empty[vs]);
      }
      if (!ok) {
        mma_commit(drain);
        drain_wait(drain, 0);
      }
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax
    const int qq = warp & 3;
    const int row = qq * 32 + lane;
    const int grow = q_tile * 128 + row;
    const uint32_t lane_base = tmem_addr(tmem_base, (uint32_t)(qq * 32), 0);
    const float sl2 = args.scale_log2;
    float m_run = -INFINITY, l_run = 0.0f;
    bool ok = true;
    for (int j = 0; j < n_kv; ++j) {
      const int b = j & 1;
      if (!mbar_wait(&s_full[b], (uint32_t)(j >> 1) & 1u, abort_v)) { ok = false; break; }
      tc_fence_after();
      uint32_t s0[32], s1[32], s2[32], s3[32];
      tmem_ld32(lane_base + (uint32_t)(b * 128 + 0), s0);
      tmem_ld32(lane_base + (uint32_t)(b * 128 + 32), s1);
      tmem_ld32(lane_base + (uint32_t)(b * 128 + 64), s2);
      tmem_ld32(lane_base + (uint32_t)(b * 128 + 96), s3);
      tmem_ld_wait(s0);
      tmem_ld_wait(s1);
      tmem_ld_wait(s2);
      tmem_ld_wait(s3);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s_empty[b]);
      float sc[128];
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        sc[c] = __uint_as_float(s0[c]);
        sc[32 + c] = __uint_as_float(s1[c]);
        sc[64 + c] = __uint_as_float(s2[c]);
        sc[96 + c] = __uint_as_float(s3[c]);
      }
      if (j == n_kv - 1) {
        const int valid = S - j * KV_TILE;
#pragma unroll
        for (int c = 0; c < 128; ++c)
          if (c >= valid) sc[c] = -INFINITY;
      }
      // eight independent partial maxima / sums (element c goes to partial
      // c % 8), combined in a fixed tree: short dependency chains, fixed order
      float mp[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) mp[e] = sc[e];
#pragma unroll
      for (int c = 8; c < 128; ++c) mp[c & 7] = fmaxf(mp[c & 7], sc[c]);
      const float mx = fmaxf(fmaxf(fmaxf(mp[0], mp[1]), fmaxf(mp[2], mp[3])),
                             fmaxf(fmaxf(mp[4], mp[5]), fmaxf(mp[6], mp[7])));
      const float m_new = fmaxf(m_run, mx * sl2);
      uint32_t pk[64];
      float sp[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int c = 0; c < 128; c += 2) {
        const float e0 = exp2f(__fmaf_rn(sc[c], sl2, -m_new));
        const float e1 = exp2f(__fmaf_rn(sc[c + 1], sl2, -m_new));
        sp[c & 7] += e0;
        sp[(c + 1) & 7] += e1;
        pk[c >> 1] = pack_bf16x2(e0, e1);
      }
      const float rs = ((sp[0] + sp[1]) + (sp[2] + sp[3])) + ((sp[4] + sp[5]) + (sp[6] + sp[7]));
      const float alpha = exp2f(m_run - m_new);
      l_run = __fmaf_rn(l_run, alpha, rs);
      if (j > 0) {
        if (!mbar_wait(o_done, (uint32_t)(j - 1) & 1u, abort_v)) { ok = false; break; }
        tc_fence_after();
        if (__any_sync(0xffffffffu, m_new > m_run)) {
#pragma unroll 1
          for (int c = 0; c < 4; ++c) {
            uint32_t o[32];
            const uint32_t ta = lane_base + 256u + (uint32_t)(c * 32);
            tmem_ld32(ta, o);
            tmem_ld_wait(o);
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tmem_st32(ta, o);
          }
          tmem_st_wait();
        }
      }
      // P_j (bf16) into the K-major 128-byte-swizzled operand tile
#pragma unroll
      for (int cc = 0; cc < 16; ++cc) {
        const uint32_t off = (uint32_t)((cc >> 3) * BOX_BYTES) + sw128_offset((uint32_t)row, (uint32_t)(cc & 7));
        *reinterpret_cast<uint4*>(sP + off) = make_uint4(pk[cc * 4], pk[cc * 4 + 1], pk[cc * 4 + 2], pk[cc * 4 + 3]);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full);
      m_run = m_new;
    }
    if (ok && mbar_wait(o_done, (uint32_t)(n_kv - 1) & 1u, abort_v)) {
      tc_fence_after();
      const float inv_l = 1.0f / l_run;
      const int HD = args.H * 128;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t o[32];
        tmem_ld32(lane_base + 256u + (uint32_t)(c * 32), o);
        tmem_ld_wait(o);
        if (grow < S && in_bounds<__nv_bfloat16>(args.o, args.o_elems,
                                                 args.o + (size_t)grow * HD + head * 128 + c * 32, 32, args.err, 12)) {
          uint4* dst = reinterpret_cast<uint4*>(args.o + (size_t)grow * HD + head * 128 + c * 32);
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            dst[g] = make_uint4(pack_bf16x2(__uint_as_float(o[g * 8 + 0]) * inv_l, __uint_as_float(o[g * 8 + 1]) * inv_l),
                                pack_bf16x2(__uint_as_float(o[g * 8 + 2]) * inv_l, __uint_as_float(o[g * 8 + 3]) * inv_l),
                                pack_bf16x2(__uint_as_float(o[g * 8 + 4]) * inv_l, __uint_as_float(o[g * 8 + 5]) * inv_l),
                                pack_bf16x2(__uint_as_float(o[g * 8 + 6]) * inv_l, __uint_as_float(o[g * 8 + 7]) * inv_l));
          }
        }
      }
      if (args.lse != nullptr && grow < S)
        if (in_bounds<float>(args.lse, args.lse_elems, args.lse + (size_t)head * S + grow, 1, args.err, 13))
          args.lse[(size_t)head * S + grow] = (m_run + log2f(l_run)) * 0.69314718055994530942f;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0 && *abort_v.flag) record_error(args.err, DEVERR_TIMEOUT);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 512);
  }
}


// ---------------------------------------------------------------------------
// Two query tiles per CTA (for long sequences): tiles A and B of one head
// share every K/V tile.  The MMA warp alternates S_A = Q_A K^T, P_A V,
// S_B = Q_B K^T, P_B V, so the tensor core works on one tile while the
// softmax warpgroup of the other runs.  TMEM: S_A [0,128), S_B [128,256),
// O_A [256,384), O_B [384,512).  The softmax writes P (bf16, two per
// column) over the first 64 columns of its S buffer and the P V product
// reads its A operand from TMEM.  Each softmax thread reads its score row
// twice (maximum, then exponentials), so it holds at most 64 scores.  O is
// rescaled only when a row maximum grows by more than 8 (base 2): the
// running maximum used for the exponent then lags the true one by at most 8,
// so probabilities before normalisation stay below 2^8; the final division
// by the running sum uses the same maximum, so the result is unchanged.
// ---------------------------------------------------------------------------
namespace {
constexpr int AT2_THREADS = 384;   // warp 0 TMA Q/K, warp 1 MMA, warp 2 TMA V, warps 4-7 tile A, 8-11 tile B
constexpr int AT2_SMEM = 1024 + TILE_BYTES * (2 + KST + VST) + 512;
constexpr float kRescaleThreshold = 8.0f;

// 16 columns of 32-bit per lane: thread t of the warp writes lane (base + t).
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

__device__ __forceinline__ void tmem_ld_wait16(uint32_t (&r)[16]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),
                 "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]),
                 "+r"(r[14]), "+r"(r[15])::"memory");
}

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// D[tmem] (+)= A[tmem] * B[smem], bf16, fp32 accumulate.
__device__ __forceinline__ void mma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
}  // namespace

__global__ void __launch_bounds__(AT2_THREADS, 1)
    attention_kernel_2q(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV, const AttnArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint8_t* sQ = smem;                       // Q_A, Q_B: 32 KB each
  uint8_t* sK = sQ + 2 * TILE_BYTES;
  uint8_t* sV = sK + KST * TILE_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sV + VST * TILE_BYTES);
  uint64_t* q_full = bars;
  uint64_t* k_full = bars + 1;
  uint64_t* k_empty = k_full + KST;
  uint64_t* v_full = k_empty + KST;
  uint64_t* v_empty = v_full + VST;
  uint64_t* s_full = v_empty + VST;    // [2]: tile A, tile B
  uint64_t* p_full = s_full + 2;       // [2]
  uint64_t* o_final = p_full + 2;      // [2]
  uint64_t* drain = o_final + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);

  griddep_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int pair = blockIdx.x, head = blockIdx.y;
  const int S = args.S;
  const int n_kv = (S + KV_TILE - 1) / KV_TILE;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < KST; ++s) { mbar_init(&k_full[s], 1); mbar_init(&k_empty[s], 1); }
    for (int s = 0; s < VST; ++s) { mbar_init(&v_full[s], 1); mbar_init(&v_empty[s], 1); }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&s_full[t], 1);
      mbar_init(&p_full[t], 4);
      mbar_init(&o_final[t], 1);
    }
    mbar_init(drain, 1);
    *abort_flag = timeout_recorded(args.err) ? 1 : 0;   // sticky timeout of an earlier launch
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  if (warp == 1) tmem_alloc(tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  griddep_wait();
  const uint32_t tmem_base = *tmem_slot;
  const WaitCtl abort_v{abort_flag, args.err, KID_ATTN_2Q};

  // a wait of an earlier launch ran out (sticky until h3_sync_check; read
  // in the prologue, beside the previous kernel): this launch skips its
  // work, before any copy or MMA is issued
  const bool skip = *abort_v.flag != 0;

  if (skip) {
  } else if (warp == 0) {
    // ------------------------------------------------------------ producer of Q and K
    if (lane == 0) {
      bool ok = true;
      int issued_k = 0;
      mbar_arrive_expect_tx(q_full, 2 * TILE_BYTES);
      for (int t = 0; t < 2; ++t) {
        tma_load_3d(sQ + t * TILE_BYTES, &tmQ, q_full, 0, head, pair * 256 + t * 128);
        tma_load_3d(sQ + t * TILE_BYTES + BOX_BYTES, &tmQ, q_full, 64, head, pair * 256 + t * 128);
      }
      for (int j = 0; j < n_kv && ok; ++j) {
        const int ks = j % KST;
        if (!mbar_wait(&k_empty[ks], ((uint32_t)(j / KST) & 1u) ^ 1u, abort_v)) { ok = false; break; }
        mbar_arrive_expect_tx(&k_full[ks], TILE_BYTES);
        tma_load_3d(sK + ks * TILE_BYTES, &tmK, &k_full[ks], 0, head, j * KV_TILE);
        tma_load_3d(sK + ks * TILE_BYTES + BOX_BYTES, &tmK, &k_full[ks], 64, head, j * KV_TILE);
        ++issued_k;
      }
      if (!ok) {
        drain_wait(q_full, 0);
        for (int j = (issued_k > KST ? issued_k - KST : 0); j < issued_k; ++j)
          drain_wait(&k_full[j % KST], (uint32_t)(j / KST) & 1u);
      }
    }
    __syncwarp();
  } else if (warp == 2) {
    // ------------------------------------------------------------ producer of V (its own thread, so a
    // V slot that frees up is refilled without waiting behind the K ring)
    if (lane == 0) {
      bool ok = true;
      int issued_v = 0;
      for (int j = 0; j < n_kv && ok; ++j) {
        const int vs = j % VST;
        if (!mbar_wait(&v_empty[vs], ((uint32_t)(j / VST) & 1u) ^ 1u, abort_v)) { ok = false; break; }
        mbar_arrive_expect_tx(&v_full[vs], TILE_BYTES);
        tma_load_3d(sV + vs * TILE_BYTES, &tmV, &v_full[vs], 0, head, j * KV_TILE);
        tma_load_3d(sV + vs * TILE_BYTES + BOX_BYTES, &tmV, &v_full[vs], 64, head, j * KV_TILE);
        ++issued_v;
      }
      if (!ok) {
        for (int j = (issued_v > VST ? issued_v - VST : 0); j < issued_v; ++j)
          drain_wait(&v_full[j % VST], (uint32_t)(j / VST) & 1u);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16(128, 128, false, false);
      constexpr uint32_t idesc_o = idesc_bf16(128, 128, false, true);   // V is MN-major
      const uint32_t q0 = smem_u32(sQ), k0 = smem_u32(sK), v0 = smem_u32(sV);
      bool ok = mbar_wait(q_full, 0, abort_v);
      // S_t = Q_t K_j^T into TMEM columns [128 t, 128 t + 128)
      auto issue_s = [&](int t, int j) {
        const uint32_t kb = k0 + (uint32_t)((j % KST) * TILE_BYTES);
        const uint32_t qb = q0 + (uint32_t)(t * TILE_BYTES);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint32_t off = (uint32_t)((k >> 2) * BOX_BYTES + (k & 3) * 32);
          mma_bf16_ss(tmem_base + (uint32_t)(t * 128), sdesc_kmajor(qb + off), sdesc_kmajor(kb + off), idesc_s,
                      k != 0 ? 1u : 0u);
        }
      };
      // O_t += P_t V_j, P_t in TMEM over S_t (16 keys = 8 columns per step)
      auto issue_pv = [&](int t, int j) {
        const uint32_t vb = v0 + (uint32_t)((j % VST) * TILE_BYTES);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint64_t b_desc = sdesc_sw128(vb + (uint32_t)(k * 2048), BOX_BYTES, 1024);
          mma_bf16_ts(tmem_base + 256u + (uint32_t)(t * 128), tmem_base + (uint32_t)(t * 128 + k * 8), b_desc,
                      idesc_o, (j | k) != 0 ? 1u : 0u);
        }
      };
      if (ok) ok = mbar_wait(&k_full[0], 0, abort_v);
      if (ok) {
        tc_fence_after();
        issue_s(0, 0);
        mma_commit(&s_full[0]);
        issue_s(1, 0);
        mma_commit(&s_full[1]);
      }
      for (int j = 0; j < n_kv && ok; ++j) {
        const bool more = j + 1 < n_kv;
        const int ks = j % KST, vs = j % VST;
        if (!mbar_wait(&v_full[vs], (uint32_t)(j / VST) & 1u, abort_v)) { ok = false; break; }
        if (more && !mbar_wait(&k_full[(j + 1) % KST], (uint32_t)((j + 1) / KST) & 1u, abort_v)) { ok = false; break; }
        for (int t = 0; t < 2; ++t) {
          if (!mbar_wait(&p_full[t], (uint32_t)j & 1u, abort_v)) { ok = false; break; }
          tc_fence_after();
          issue_pv(t, j);
          if (more) issue_s(t, j + 1);     // overwrites S_t / P_t after P_t V_j (in order)
          if (t == 1) {
            mma_commit(&k_empty[ks]);
            mma_commit(&v_empty[vs]);
          }
          mma_commit(more ? &s_full[t] : &o_final[t]);
        }
      }
      if (!ok) {
        mma_commit(drain);
        drain_wait(drain, 0);
      }
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax
    const int t = (warp - 4) >> 2;             // query tile A (0) or B (1)
    const int qq = warp & 3;
    const int row = qq * 32 + lane;
    const int grow = pair * 256 + t * 128 + row;
    const uint32_t s_base = tmem_addr(tmem_base, (uint32_t)(qq * 32), (uint32_t)(t * 128));
    const uint32_t o_base = s_base + 256u;
    const float sl2 = args.scale_log2;
    float m_used = -INFINITY, l_run = 0.0f;
    bool ok = true;
    for (int j = 0; j < n_kv; ++j) {
      if (!mbar_wait(&s_full[t], (uint32_t)j & 1u, abort_v)) { ok = false; break; }
      tc_fence_after();
      const int valid = S - j * KV_TILE;     // keys of this tile that exist (>= 1)
      // all 128 scores of the row, requested before one wait and kept in
      // registers for both passes (keys past the end of the sequence are set
      // to -inf: they take no part in the maximum and get probability 0)
      uint32_t r[4][32];
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) tmem_ld32(s_base + (uint32_t)(q4 * 32), r[q4]);
      tmem_ld_wait(r[0]);
      if (valid < KV_TILE) {
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4)
#pragma unroll
          for (int c = 0; c < 32; ++c)
            if (q4 * 32 + c >= valid) r[q4][c] = __float_as_uint(-INFINITY);
      }
      // pass 1: row maximum, eight independent partial maxima (fixed
      // combination order)
      float mp[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) mp[e] = -INFINITY;
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4)
#pragma unroll
        for (int c = 0; c < 32; ++c) mp[c & 7] = fmaxf(mp[c & 7], __uint_as_float(r[q4][c]));
      const float mx = fmaxf(fmaxf(fmaxf(mp[0], mp[1]), fmaxf(mp[2], mp[3])),
                             fmaxf(fmaxf(mp[4], mp[5]), fmaxf(mp[6], mp[7])));
      const float m_tile = mx * sl2;
      // lazy rescale: move the running maximum only when it grows by > 8
      const bool need = m_tile > m_used + kRescaleThreshold;
      if (__any_sync(0xffffffffu, need)) {
        const float m_new = need ? fmaxf(m_tile, m_used) : m_used;
        const float alpha = ex2_approx(m_used - m_new);   // 0 when m_used = -inf
        l_run *= alpha;
        if (j > 0) {
          // O_t is final for tiles < j (the S_t(j) commit covers P_t V_{j-1});
          // 16 columns at a time, as the row's scores stay in registers
#pragma unroll 1
          for (int c = 0; c < 8; ++c) {
            uint32_t o[16];
            tmem_ld16(o_base + (uint32_t)(c * 16), o);
            tmem_ld_wait16(o);
#pragma unroll
            for (int e = 0; e < 16; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tmem_st16(o_base + (uint32_t)(c * 16), o);
          }
        }
        m_used = m_new;
      }
      // pass 2: P = 2^(s * scale_log2 - m_used) as bf16 over the S columns,
      // two keys per packed fp32 FMA; eight partial sums (as float pairs)
      const float2 sl2x2 = make_float2(sl2, sl2);
      const float2 negm = make_float2(-m_used, -m_used);
      float2 sp[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) sp[e] = make_float2(0.0f, 0.0f);
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        uint32_t pk[16];
#pragma unroll
        for (int c = 0; c < 16; ++c) {         // keys 32 q4 + 2c and 32 q4 + 2c + 1
          const float2 z = __ffma2_rn(make_float2(__uint_as_float(r[q4][2 * c]), __uint_as_float(r[q4][2 * c + 1])),
                                      sl2x2, negm);
          const float e0 = ex2_approx(z.x), e1 = ex2_approx(z.y);
          sp[c & 3] = __fadd2_rn(sp[c & 3], make_float2(e0, e1));
          pk[c] = pack_bf16x2(e0, e1);
        }
        // keys [32 q4, 32 q4 + 32) -> packed columns [16 q4, 16 q4 + 16):
        // their scores are already in registers
        tmem_st16(s_base + (uint32_t)(q4 * 16), pk);
      }
      l_run += ((sp[0].x + sp[0].y) + (sp[1].x + sp[1].y)) + ((sp[2].x + sp[2].y) + (sp[3].x + sp[3].y));
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[t]);
    }
    if (ok && mbar_wait(&o_final[t], 0, abort_v)) {
      tc_fence_after();
      const float inv_l = 1.0f / l_run;
      const int HD = args.H * 128;
      // The normalised rows go out through the K ring, idle now (the
      // o_final commit covers every S MMA, and no K load is left in flight):
      // each warp stages its 32 rows x 128 channels (8 KB, 16-byte unit u of
      // row r at unit u ^ (r & 7)), then two rows per store instruction
      // leave as whole lines.
      uint8_t* stg = sK + (size_t)(warp - 4) * 8192;
      const int grow0 = grow - lane;
      const bool row_ok = grow < S && in_bounds<__nv_bfloat16>(args.o, args.o_elems,
                                                               args.o + (size_t)grow * HD + head * 128, 128, args.err,
                                                               12);
      const unsigned ok_rows = __ballot_sync(0xffffffffu, row_ok);
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t o[32];
        tmem_ld32(o_base + (uint32_t)(c * 32), o);
        tmem_ld_wait(o);
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          const int u = c * 4 + g;
          *reinterpret_cast<uint4*>(stg + lane * 256 + ((u ^ (lane & 7)) << 4)) =
              make_uint4(pack_bf16x2(__uint_as_float(o[g * 8 + 0]) * inv_l, __uint_as_float(o[g * 8 + 1]) * inv_l),
                         pack_bf16x2(__uint_as_float(o[g * 8 + 2]) * inv_l, __uint_as_float(o[g * 8 + 3]) * inv_l),
                         pack_bf16x2(__uint_as_float(o[g * 8 + 4]) * inv_l, __uint_as_float(o[g * 8 + 5]) * inv_l),
                         pack_bf16x2(__uint_as_float(o[g * 8 + 6]) * inv_l, __uint_as_float(o[g * 8 + 7]) * inv_l));
        }
      }
      __syncwarp();
#pragma unroll 4
      for (int it = 0; it < 16; ++it) {
        const int r = it * 2 + (lane >> 4), u = lane & 15;
        if ((ok_rows >> r) & 1u)
          *reinterpret_cast<uint4*>(args.o + (size_t)(grow0 + r) * HD + head * 128 + u * 8) =
              *reinterpret_cast<const uint4*>(stg + r * 256 + ((u ^ (r & 7)) << 4));
      }
      if (args.lse != nullptr && grow < S)
        if (in_bounds<float>(args.lse, args.lse_elems, args.lse + (size_t)head * S + grow, 1, args.err, 13))
          args.lse[(size_t)head * S + grow] = (m_used + log2f(l_run)) * 0.69314718055994530942f;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0 && *abort_v.flag) record_error(args.err, DEVERR_TIMEOUT);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 512);
  }
}

// Two query tiles per CTA (measured faster at every length down to 505
// rows); H3_ATTN_QTILES=1 in the environment selects the one-tile kernel
// (tests cover both).
//
// A grid of one wave or less starts in plain stream order, not early beside
// the kernel before it.  Measured with per-CTA clock stamps at 505 rows (112
// CTAs): CTAs that started early and passed griddepcontrol.wait when the QKV
// GEMM ended lived 19 us against 11.6 us.  The extra time fell on the code
// that each CTA runs first (the first softmax step, the masked last one, the
// output stores) and on the first MMAs.  The middle softmax steps ran at the
// same speed either way.  The block took 368 instead of 374 us.  At three
// waves (1824 rows) only the first wave starts early, and the two launch
// modes measured the same.
cudaError_t launch_attention(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                             const AttnArgs& a, cudaStream_t stream) {
  int qtiles = 2;
  if (const char* env = getenv("H3_ATTN_QTILES")) {
    const int f = atoi(env);
    if (f == 1 || f == 2) qtiles = f;
  }
  const long long ctas = (long long)(qtiles == 2 ? (a.S + 255) / 256 : (a.S + 127) / 128) * a.H;
  const bool early = ctas > num_sms();
  static_assert(tmem_footprint_exclusive(AT_SMEM) && tmem_footprint_exclusive(AT2_SMEM),
                "an attention CTA must hold its SM's TMEM alone");
  if (!tmem_exclusive(qtiles == 2 ? AT2_SMEM : AT_SMEM)) return cudaErrorNotSupported;
  cudaError_t e;
  if (qtiles == 2) {
    e = cudaFuncSetAttribute(attention_kernel_2q, cudaFuncAttributeMaxDynamicSharedMemorySize, AT2_SMEM);
    if (e != cudaSuccess) return e;
    const dim3 grid((unsigned)((a.S + 255) / 256), (unsigned)a.H);
    e = launch_kernel_ex(attention_kernel_2q, grid, dim3(AT2_THREADS), AT2_SMEM, stream, 1, early, tmQ, tmK, tmV, a);
    if (e != cudaSuccess) return e;
    set_kernel_info("attention_kernel_2q tcgen05.mma.cta_group::1.kind::f16 q_tiles=2x128 kv_tile=128 "
                    "k_stages=%d v_stages=%d acc=f32 tmem=S_A,S_B,O_A,O_B P-in-TMEM lazy-rescale=%g grid=%ux%u "
                    "early-start=%d",
                    KST, VST, (double)kRescaleThreshold, grid.x, grid.y, early ? 1 : 0);
  } else {
    e = cudaFuncSetAttribute(attention_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, AT_SMEM);
    if (e != cudaSuccess) return e;
    const dim3 grid((unsigned)((a.S + 127) / 128), (unsigned)a.H);
    e = launch_kernel_ex(attention_kernel, grid, dim3(AT_THREADS), AT_SMEM, stream, 1, early, tmQ, tmK, tmV, a);
    if (e != cudaSuccess) return e;
    set_kernel_info("attention_kernel tcgen05.mma.cta_group::1.kind::f16 q_tile=128 kv_tile=128 k_stages=%d "
                    "v_stages=%d acc=f32 tmem=S0,S1,O softmax=fp32-online grid=%ux%u early-start=%d",
                    KST, VST, grid.x, grid.y, early ? 1 : 0);
  }
  return cudaGetLastError();
}

}  // namespace h3
