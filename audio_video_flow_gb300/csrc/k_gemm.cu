// tcgen05 GEMMs for the H3 block projections.
//
// gemm_bf16_tc<EPI, BN>: D[256 x BN] tiles of act[M][K] . W[rows][K]^T, bf16
// in, fp32 accumulate in TMEM, with the epilogue fused per projection:
//   EPI_PLAIN   y = bf16(acc + b)
//   EPI_QKV     q and k columns of a head: per-head Q/K RMSNorm, then the
//               partial three-axis MM-RoPE on 96 of the 128 channels (RFC
//               section 4: norm before RoPE); v columns plain
//   EPI_RESID   y = bf16(x + gate[r] * bf16(acc + b))   (RFC s4 residual order)
//   EPI_SWIGLU  a = bf16(SiLU(g) * u) with g, u the paired gate / value tiles
//               (the h3-metal README, section "Metal 4 and TensorOps paths",
//               pairs the FC1 gate and up tiles so SwiGLU happens before the
//               store)
// Structure: persistent CTA pairs (clusters of two, one CTA per SM), static
// grouped tile order (see tile_coords).  A pair owns a 256 x BN tile: each CTA
// stages its 128 rows of A and half (BN/2) of the tile's weight rows, and one
// thread of the even CTA issues tcgen05.mma.cta_group::2 (M = 256), which
// reads both CTAs' shared memory and accumulates each CTA's 128 rows in its
// own TMEM.  Per SM this moves 32 KB of operands per 64-deep k-block instead
// of the 48 KB a 128 x 256 tile on one SM needs, and leaves room for a deeper
// ring (6-8 stages).  Warp 0 of each CTA issues its TMA loads (completion
// counted on the even CTA's barrier) and, above 16 row tiles, L2 prefetches
// of the weights further ahead; warp 1 of the even CTA issues the MMAs into
// one of two TMEM accumulators (2 x BN columns) and releases ring stages to
// both CTAs with a multicast tcgen05.commit; warps 2-9 of each CTA drain the other accumulator through
// tcgen05.ld and run the epilogue, two warps per TMEM lane quadrant (warp w
// reads lanes 32 (w % 4) ..), warps 2-5 on the first and 6-9 on the second
// half of the tile's columns.  BN (256, 192 or 128) is chosen per launch to
// fill the SMs; it changes the tiling, never the reduction: with whole tiles
// every output element is the same fixed sequence of 16-deep MMAs over K, so
// the result does not depend on M, BN or the grid.  Stream-K launches (the
// residual GEMMs of a block when whole tiles would leave pairs idle) add
// fp32 partial sums of k-ranges in a fixed order.
//
// adaln_table_kernel: the AdaLN projection.  Its M dimension is only T <= 16
// timestep rows, so the GEMM runs transposed: the 18*D weight rows are the
// 128-row M operand streamed by TMA (two 64-column boxes per stage, 256
// contiguous bytes of every row), and u = bf16(SiLU(t_cond)), written once by
// silu_rows_kernel and TMA-loaded into shared memory by every CTA, is the
// resident N = 16 operand.  The kernel is bound by the weight stream from HBM.
#include "h3_device.cuh"

#include "h3_internal.h"

#include <cstdio>
#include <cstdlib>

namespace h3 {

namespace {

constexpr int BM = 128, BK = 64;
constexpr int A_STAGE_BYTES = BM * BK * 2;   // 16 KB
constexpr int GEMM_THREADS = 320;   // producer, MMA issuer, 8 epilogue warps

// Per CTA of a pair: its 128 rows of A and BN/2 rows of B per 64-deep k-block.
template <int BN>
struct GemmCfg {
  static constexpr int B_ROWS = BN / 2;
  static constexpr int B_STAGE_BYTES = B_ROWS * BK * 2;
  static constexpr int STAGE_BYTES = A_STAGE_BYTES + B_STAGE_BYTES;
  static constexpr int STAGES = (196608 / STAGE_BYTES) > 8 ? 8 : (196608 / STAGE_BYTES);   // 6, 7, 8
  static constexpr int SMEM = 1024 + STAGES * STAGE_BYTES + 256;
};

// The gated-residual, SwiGLU and QKV epilogues of 256-wide tiles stage each
// epilogue warp's 32 rows x 64 columns (bf16, 4 KB) in shared memory after
// the barriers, so that their global loads and stores move whole 128-byte
// lines.
constexpr int EPI_STAGE_WARP_BYTES = 32 * 128;
constexpr int EPI_STAGE_BYTES = 8 * EPI_STAGE_WARP_BYTES;
template <int EPI, int BN>
__host__ __device__ constexpr bool gemm_staged_epi() {
  return BN == 256 && (EPI == EPI_RESID || EPI == EPI_SWIGLU || EPI == EPI_QKV);
}
template <int EPI, int BN>
__host__ __device__ constexpr int gemm_smem() {
  return GemmCfg<BN>::SMEM + (gemm_staged_epi<EPI, BN>() ? EPI_STAGE_BYTES : 0);
}
static_assert(gemm_smem<EPI_RESID, 256>() <= 232448, "the staged epilogue fits the shared-memory limit");

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

__device__ __forceinline__ void tma_prefetch_l2(const CUtensorMap* tm, int32_t x, int32_t y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global [%0, {%1, %2}];" ::"l"(reinterpret_cast<uint64_t>(tm)),
               "r"(x), "r"(y)
               : "memory");
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

// Columns [n0, n0 + w) of tile n_blk (plain and residual epilogues; the
// others always use uniform BN-wide tiles).
struct NTile {
  int n0, w;
};
template <int EPI, int BN>
__device__ __forceinline__ NTile n_tile(const GemmArgs& a, int n_blk) {
  if ((EPI != EPI_PLAIN && EPI != EPI_RESID) || a.nw1 == 0) return {n_blk * BN, BN};
  if (n_blk < a.ncnt1) return {n_blk * a.nw1, a.nw1};
  return {a.ncnt1 * a.nw1 + (n_blk - a.ncnt1) * a.nw2, a.nw2};
}

// First weight row of the B rows that CTA `rank` of the pair loads for tile
// n_blk.  The tile's N columns are rank 0's rows then rank 1's rows.
template <int EPI, int BN>
__device__ __forceinline__ int b_tile_row(const GemmArgs& a, int n_blk, uint32_t rank) {
  if (EPI == EPI_SWIGLU) return (rank ? a.F : 0) + n_blk * 128;            // gate rows | value rows
  if (EPI == EPI_QKV && BN == 256) {
    if (n_blk < a.H) return n_blk * 384 + (int)rank * 128;                  // q | k of head n_blk
    const int p = n_blk - a.H;
    return (2 * p + (int)rank) * 384 + 256;                                 // v of heads 2p | 2p+1
  }
  if (EPI == EPI_QKV) return (n_blk / 3) * 384 + (n_blk % 3) * 128 + (int)rank * 64;   // q, k or v of a head
  const NTile t = n_tile<EPI, BN>(a, n_blk);
  return t.n0 + (int)rank * (t.w / 2);
}

// Tile order (tiles of 256 rows, one per CTA pair): groups of GROUP_M
// m-tiles; inside a group m runs fastest, then n.  The CTAs running at one time then share a few weight tiles and a group
// of activation rows that both stay in L2 (with m fastest over all of M, a
// tall activation matrix would be streamed from HBM once per weight column).
constexpr int GROUP_M = 16;
__device__ __forceinline__ void tile_coords(int tile, int num_m, int num_n, int& m_blk, int& n_blk) {
  const int per_group = GROUP_M * num_n;
  const int g = tile / per_group;
  const int m0 = g * GROUP_M;
  const int gm = num_m - m0 < GROUP_M ? num_m - m0 : GROUP_M;
  const int r = tile - g * per_group;
  m_blk = m0 + r % gm;
  n_blk = r / gm;
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

// Columns [n0, n0 + w) of the tile, w a multiple of 16: 32-column chunks and
// at most one 16-column tail.
template <int NC>
__device__ __forceinline__ void tmem_ld_chunk(uint32_t taddr, uint32_t (&r)[32]) {
  if (NC == 32) {
    tmem_ld32(taddr, r);
    tmem_ld_wait(r);
  } else {
    uint32_t h[16];
    tmem_ld16(taddr, h);
    tmem_ld_wait16(h);
#pragma unroll
    for (int i = 0; i < 16; ++i) r[i] = h[i];
  }
}

// bounds-checked build: n output elements at p inside the output buffer
__device__ __forceinline__ bool out_ok(const GemmArgs& a, const __nv_bfloat16* p, int n, uint32_t site) {
  return in_bounds<__nv_bfloat16>(a.out, a.out_elems, p, (size_t)n, a.err, site);
}

template <int NC>
__device__ __forceinline__ void plain_chunk(const GemmArgs& a, uint32_t tc, int m, bool valid, int n0) {
  uint32_t r[32];
  tmem_ld_chunk<NC>(tc, r);
  if (valid) {
    __nv_bfloat16* dst = a.out + (size_t)m * a.ldo + n0;
#pragma unroll
    for (int g = 0; g < NC / 8; ++g) {
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
        if (out_ok(a, dst + g * 8, 8, 1)) *reinterpret_cast<uint4*>(dst + g * 8) = w;
      }
    }
  }
}

// Column half `half` of a w-column tile: the first half takes the first
// floor(w / 64) 32-column chunks, the second the other chunks and the
// 16-column tail.
__device__ __forceinline__ void half_range(int w, int half, int& c0, int& c1) {
  const int mid = ((w >> 5) >> 1) << 5;
  c0 = half ? mid : 0;
  c1 = half ? w : mid;
}

__device__ __forceinline__ void epi_plain(const GemmArgs& a, uint32_t tacc, int m, bool valid, NTile t, int half) {
  int c, c1;
  half_range(t.w, half, c, c1);
#pragma unroll 1
  for (; c + 32 <= c1; c += 32) plain_chunk<32>(a, tacc + c, m, valid, t.n0 + c);
  if (c < c1) plain_chunk<16>(a, tacc + c, m, valid, t.n0 + c);
}

__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_u32(uint32_t* p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

template <int NC>
__device__ __forceinline__ void resid_chunk(const GemmArgs& a, uint32_t tc, int m, bool valid,
                                            const __nv_bfloat16* gate, int n0, float& ss) {
  uint32_t r[32];
  tmem_ld_chunk<NC>(tc, r);
  if (valid && n0 < a.n_valid &&
      in_bounds<__nv_bfloat16>(a.resid, a.resid_elems, a.resid + (size_t)m * a.ldr + n0, NC, a.err, 2) &&
      in_bounds<__nv_bfloat16>(a.table, a.table_elems, gate + n0, NC, a.err, 3) &&
      out_ok(a, a.out + (size_t)m * a.ldo + n0, NC, 4)) {
    const uint4* xs = reinterpret_cast<const uint4*>(a.resid + (size_t)m * a.ldr + n0);
    const uint4* gs = reinterpret_cast<const uint4*>(gate + n0);
    uint4* dst = reinterpret_cast<uint4*>(a.out + (size_t)m * a.ldo + n0);
#pragma unroll
    for (int g = 0; g < NC / 8; ++g) {
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
        ss = __fmaf_rn(bf16_lo(ow[e]), bf16_lo(ow[e]), ss);
        ss = __fmaf_rn(bf16_hi(ow[e]), bf16_hi(ow[e]), ss);
      }
      dst[g] = make_uint4(ow[0], ow[1], ow[2], ow[3]);
    }
  }
}

__device__ __forceinline__ void epi_resid(const GemmArgs& a, uint32_t tacc, int m, bool valid, NTile t, int half,
                                          int n_blk) {
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
  int c, c1;
  half_range(t.w, half, c, c1);
  float ss = 0.0f;
#pragma unroll 1
  for (; c + 32 <= c1; c += 32) resid_chunk<32>(a, tacc + c, m, valid, gate, t.n0 + c, ss);
  if (c < c1) resid_chunk<16>(a, tacc + c, m, valid, gate, t.n0 + c, ss);
  if (a.nrm_h && m < a.M) a.nrm_part[(size_t)(2 * n_blk + half) * (a.num_m * 256) + m] = ss;
}

// The residual and gate rows of this warp's row and column half, asked
// into L1 ahead of the epilogue (each lane its own row, 128-byte lines): the
// owner of a stream-K tile issues them before it waits for the partials, so
// the epilogue's loads hit L1 instead of paying an L2 round trip per chunk.
__device__ __forceinline__ void prefetch_l1(const void* p) {
  asm volatile("prefetch.global.L1 [%0];" ::"l"(p));
}
__device__ __forceinline__ void epi_resid_prefetch(const GemmArgs& a, int m, NTile t, int half) {
  if (m >= a.M) return;
  const int tg = a.tag[m], ti = a.tidx[m];
  if ((unsigned)tg > 2u || (unsigned)ti >= (unsigned)a.T) return;   // reported by the epilogue
  const __nv_bfloat16* gate = a.table + ((size_t)(ti * 3 + tg) * 6 + a.chunk) * a.D;
  int c, c1;
  half_range(t.w, half, c, c1);
  for (; c < c1; c += 64) {
    const int n0 = t.n0 + c;
    if (n0 >= a.n_valid) break;
    prefetch_l1(a.resid + (size_t)m * a.ldr + n0);
    prefetch_l1(gate + n0);
  }
}

// Unit u (16 bytes) of row r of a warp's staging buffer (32 rows x 128
// bytes) sits at unit u ^ (r & 7): one row per lane and eight lanes per row
// both reach all 32 banks without conflict.
__device__ __forceinline__ uint4* stage_unit(uint8_t* buf, int r, int u) {
  return reinterpret_cast<uint4*>(buf + r * 128 + ((u ^ (r & 7)) << 4));
}

// The gated residual through the warp's staging buffer, 64 columns at a
// time: the warp reads the residual rows as whole lines (eight lanes per row,
// four rows per load), each lane combines its own row with its accumulator
// row and gate exactly as resid_chunk does, and the warp writes the output
// rows as whole lines.  Rows whose metadata is out of range are left
// unwritten (their lanes vote them out).  Columns past the last full 64 go
// through resid_chunk.
__device__ __forceinline__ void epi_resid_staged(const GemmArgs& a, uint32_t tacc, int m, bool valid, NTile t,
                                                 int half, int n_blk, uint8_t* buf) {
  const int lane = (int)(threadIdx.x & 31u);
  const int row0 = m - lane;
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
  int c, c1;
  half_range(t.w, half, c, c1);
  float ss = 0.0f;
#pragma unroll 1
  for (; c + 64 <= c1 && t.n0 + c + 64 <= a.n_valid; c += 64) {
    const int n0 = t.n0 + c;
#pragma unroll
    for (int it = 0; it < 8; ++it) {
      const int r = it * 4 + (lane >> 3), u = lane & 7, gm = row0 + r;
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      const __nv_bfloat16* src = a.resid + (size_t)gm * a.ldr + n0 + u * 8;
      if (gm < a.M && in_bounds<__nv_bfloat16>(a.resid, a.resid_elems, src, 8, a.err, 2))
        v = *reinterpret_cast<const uint4*>(src);
      *stage_unit(buf, r, u) = v;
    }
    uint32_t r0[32], r1[32];
    tmem_ld32(tacc + c, r0);
    tmem_ld_wait(r0);
    tmem_ld32(tacc + c + 32, r1);
    tmem_ld_wait(r1);
    const bool ok = valid && in_bounds<__nv_bfloat16>(a.table, a.table_elems, gate + n0, 64, a.err, 3);
    const unsigned ok_rows = __ballot_sync(0xffffffffu, ok);
    __syncwarp();
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      uint4 ov = make_uint4(0u, 0u, 0u, 0u);
      if (ok) {
        const uint4 xv = *stage_unit(buf, lane, u);
        const uint4 gv = *reinterpret_cast<const uint4*>(gate + n0 + u * 8);
        const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
        const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w};
        uint32_t ow[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int j = u * 8 + 2 * e;   // column of the 64
          const uint32_t acc_lo = j < 32 ? r0[j] : r1[j - 32];
          const uint32_t acc_hi = j < 32 ? r0[j + 1] : r1[j - 31];
          const float flo = bf16_round(__uint_as_float(acc_lo) + bias_at(a.bias, n0 + j));
          const float fhi = bf16_round(__uint_as_float(acc_hi) + bias_at(a.bias, n0 + j + 1));
          const float ylo = __fmaf_rn(bf16_lo(gw[e]), flo, bf16_lo(xw[e]));
          const float yhi = __fmaf_rn(bf16_hi(gw[e]), fhi, bf16_hi(xw[e]));
          ow[e] = pack_bf16x2(ylo, yhi);
          ss = __fmaf_rn(bf16_lo(ow[e]), bf16_lo(ow[e]), ss);
          ss = __fmaf_rn(bf16_hi(ow[e]), bf16_hi(ow[e]), ss);
        }
        ov = make_uint4(ow[0], ow[1], ow[2], ow[3]);
      }
      *stage_unit(buf, lane, u) = ov;
    }
    __syncwarp();
#pragma unroll
    for (int it = 0; it < 8; ++it) {
      const int r = it * 4 + (lane >> 3), u = lane & 7, gm = row0 + r;
      __nv_bfloat16* dst = a.out + (size_t)gm * a.ldo + n0 + u * 8;
      if (((ok_rows >> r) & 1u) && out_ok(a, dst, 8, 4)) *reinterpret_cast<uint4*>(dst) = *stage_unit(buf, r, u);
    }
    __syncwarp();
  }
#pragma unroll 1
  for (; c + 32 <= c1; c += 32) resid_chunk<32>(a, tacc + c, m, valid, gate, t.n0 + c, ss);
  if (c < c1) resid_chunk<16>(a, tacc + c, m, valid, gate, t.n0 + c, ss);
  if (a.nrm_h && m < a.M) a.nrm_part[(size_t)(2 * n_blk + half) * (a.num_m * 256) + m] = ss;
}

// SwiGLU: gate columns g and value columns u of the tile (128 each; column
// half `half` takes output columns 64 half .. 64 half + 63), out =
// SiLU(bf16(g + b_g)) * bf16(u + b_u).  The 64 outputs of this lane's row go
// to its row of the warp's staging buffer, then the warp writes the 32 rows
// as whole lines.
__device__ __forceinline__ void epi_swiglu_staged(const GemmArgs& a, uint32_t tacc, int m, bool valid, int n_blk,
                                                  int half, uint8_t* buf) {
  const int lane = (int)(threadIdx.x & 31u);
  const int row0 = m - lane;
  const int n0 = n_blk * 128 + half * 64;   // the half's first output column
  const bool ok = valid && out_ok(a, a.out + (size_t)m * a.ldo + n0, 64, 5);
  const unsigned ok_rows = __ballot_sync(0xffffffffu, ok);
#pragma unroll 1
  for (int cc = 0; cc < 2; ++cc) {
    const int c = 2 * half + cc;
    uint32_t g[32], u[32];
    tmem_ld32(tacc + c * 32, g);
    tmem_ld32(tacc + 128 + c * 32, u);
    tmem_ld_wait(g);
    tmem_ld_wait(u);
    float v[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const float gv = bf16_round(__uint_as_float(g[j]) + bias_at(a.bias, n0 + cc * 32 + j));
      const float uv = bf16_round(__uint_as_float(u[j]) + bias_at(a.bias, a.F + n0 + cc * 32 + j));
      v[j] = ok ? (gv / (1.0f + expf(-gv))) * uv : 0.0f;
    }
#pragma unroll
    for (int k = 0; k < 4; ++k)
      *stage_unit(buf, lane, cc * 4 + k) =
          make_uint4(pack_bf16x2(v[8 * k + 0], v[8 * k + 1]), pack_bf16x2(v[8 * k + 2], v[8 * k + 3]),
                     pack_bf16x2(v[8 * k + 4], v[8 * k + 5]), pack_bf16x2(v[8 * k + 6], v[8 * k + 7]));
  }
  __syncwarp();
#pragma unroll
  for (int it = 0; it < 8; ++it) {
    const int r = it * 4 + (lane >> 3), un = lane & 7;
    if ((ok_rows >> r) & 1u)
      *reinterpret_cast<uint4*>(a.out + (size_t)(row0 + r) * a.ldo + n0 + un * 8) = *stage_unit(buf, r, un);
  }
  __syncwarp();
}

// The fused RMSNorm + modulation of one owned tile's column half for the 32
// rows of this warp (see GemmArgs::nrm_h): waits until every owner warp of
// the row tile has stored its partial sums; lane l then adds row (row0 + l)'s
// partials in column order, and the warp walks the 32 rows with lane l on
// columns 4l..4l+3 of the half (coalesced 8-byte loads and stores).
__device__ __forceinline__ bool fused_norm(const GemmArgs& a, int m_blk, int n_blk, int row0, int half, int lane,
                                           const WaitCtl& c) {
  const uint32_t* cnt = a.nrm_cnt + m_blk;
  if (ld_acquire_u32(cnt) < a.nrm_target) {
    const uint64_t t0 = globaltimer();
    for (uint32_t i = 1;; ++i) {
      if (ld_acquire_u32(cnt) >= a.nrm_target) break;
      if ((i & 31u) == 0 && wait_gives_up(c, t0, kSiteNormCount)) return false;
    }
  }
  const int m = row0 + lane;
  int trow = -1;
  float inv = 0.0f;
  if (m < a.M) {
    const int tg = a.tag[m], ti = a.tidx[m];
    if ((unsigned)tg <= 2u && (unsigned)ti < (unsigned)a.T) {   // bad rows are reported by the epilogue
      trow = ti * 3 + tg;
      const int mp = a.num_m * 256;
      float ss = 0.0f;
      for (int j = 0; j < 2 * a.num_n; ++j) ss += a.nrm_part[(size_t)j * mp + m];
      inv = 1.0f / sqrtf(ss / (float)a.D + a.eps);
    }
  }
  const NTile t = n_tile<EPI_RESID, 256>(a, n_blk);
  int c0, c1;
  half_range(t.w, half, c0, c1);
  const int n = t.n0 + c0 + 4 * lane;
  const bool on = 4 * lane < c1 - c0 && n < a.n_valid;
  uint2 gv = make_uint2(0u, 0u);
  if (on) gv = *reinterpret_cast<const uint2*>(a.nrm_gain + n);
#pragma unroll 4
  for (int r = 0; r < 32; ++r) {
    const int tr = __shfl_sync(0xffffffffu, trow, r);
    const float iv = __shfl_sync(0xffffffffu, inv, r);
    if (tr < 0 || !on) continue;
    const size_t mr = (size_t)(row0 + r);
    const __nv_bfloat16* trp = a.table + (size_t)tr * 6 * a.D;
    const uint2 xv = *reinterpret_cast<const uint2*>(a.out + mr * a.ldo + n);
    const uint2 hv = *reinterpret_cast<const uint2*>(trp + (size_t)a.nrm_shift * a.D + n);
    const uint2 sv = *reinterpret_cast<const uint2*>(trp + (size_t)a.nrm_scale * a.D + n);
    const uint32_t xw[2] = {xv.x, xv.y}, gw[2] = {gv.x, gv.y}, hw[2] = {hv.x, hv.y}, sw[2] = {sv.x, sv.y};
    uint32_t ow[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const float nlo = (bf16_lo(xw[e]) * iv) * bf16_lo(gw[e]);
      const float nhi = (bf16_hi(xw[e]) * iv) * bf16_hi(gw[e]);
      ow[e] = pack_bf16x2(__fmaf_rn(nlo, 1.0f + bf16_lo(sw[e]), bf16_lo(hw[e])),
                          __fmaf_rn(nhi, 1.0f + bf16_hi(sw[e]), bf16_hi(hw[e])));
    }
    *reinterpret_cast<uint2*>(a.nrm_h + mr * a.D + n) = make_uint2(ow[0], ow[1]);
  }
  return true;
}

// Q or K columns of head h (128 accumulator columns at tpart): per-head
// RMSNorm of the bf16-cast projection, then the rotation of channels 0..95
// (channel j < 48 with j + 48, band j/16 = t, h, w), channels 96..127 normed only.
__device__ __forceinline__ void epi_qk_part(const GemmArgs& a, uint32_t tpart, int m, bool valid, int h,
                                            int part, const float (&pos)[3]) {
  const int cb = h * 384 + part * 128;       // output / weight column of channel 0
  const __nv_bfloat16* gain = part ? a.k_gain : a.q_gain;
  float ss = 0.f;
#pragma unroll 1
  for (int c = 0; c < 4; ++c) {
    uint32_t r[32];
    tmem_ld32(tpart + c * 32, r);
    tmem_ld_wait(r);
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const float v = bf16_round(__uint_as_float(r[j]) + bias_at(a.bias, cb + c * 32 + j));
      ss = __fmaf_rn(v, v, ss);
    }
  }
  const float inv = 1.0f / sqrtf(ss * (1.0f / 128.0f) + a.eps);
#pragma unroll 1
  for (int band = 0; band < 3; ++band) {
    const float p = band == 0 ? pos[0] : (band == 1 ? pos[1] : pos[2]);
    uint32_t lo[16], hi[16];
    tmem_ld16(tpart + band * 16, lo);
    tmem_ld16(tpart + 48 + band * 16, hi);
    tmem_ld_wait(lo, hi);
    if (valid) {
      float o1[16], o2[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int j = band * 16 + i;
        float sn, cs;
        sincosf(p * a.omega[i], &sn, &cs);
        const float v1 = bf16_round(__uint_as_float(lo[i]) + bias_at(a.bias, cb + j));
        const float v2 = bf16_round(__uint_as_float(hi[i]) + bias_at(a.bias, cb + 48 + j));
        const float x1 = bf16_round(v1 * inv * __bfloat162float(gain[j]));
        const float x2 = bf16_round(v2 * inv * __bfloat162float(gain[48 + j]));
        o1[i] = __fmaf_rn(x1, cs, -(x2 * sn));
        o2[i] = __fmaf_rn(x2, cs, x1 * sn);
      }
      __nv_bfloat16* dst = a.out + (size_t)m * a.ldo + cb;
      if (out_ok(a, dst + band * 16, 16, 6)) store16_bf16(dst + band * 16, o1);
      if (out_ok(a, dst + 48 + band * 16, 16, 7)) store16_bf16(dst + 48 + band * 16, o2);
    }
  }
  uint32_t r[32];
  tmem_ld32(tpart + 96, r);
  tmem_ld_wait(r);
  if (valid) {
    float v[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const float x = bf16_round(__uint_as_float(r[j]) + bias_at(a.bias, cb + 96 + j));
      v[j] = x * inv * __bfloat162float(gain[96 + j]);
    }
    if (out_ok(a, a.out + (size_t)m * a.ldo + cb + 96, 32, 8)) store32_bf16(a.out + (size_t)m * a.ldo + cb + 96, v);
  }
}

// V columns of one head (128 accumulator columns at tpart).
__device__ __forceinline__ void epi_v_head(const GemmArgs& a, uint32_t tpart, int m, bool valid, int head) {
#pragma unroll 1
  for (int c = 0; c < 4; ++c) {
    uint32_t r[32];
    tmem_ld32(tpart + c * 32, r);
    tmem_ld_wait(r);
    if (valid && head < a.H) {
      const int cb = head * 384 + 256 + c * 32;
      float v[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]) + bias_at(a.bias, cb + j);
      if (out_ok(a, a.out + (size_t)m * a.ldo + cb, 32, 9)) store32_bf16(a.out + (size_t)m * a.ldo + cb, v);
    }
  }
}

// The warp's staged 64 columns of its 32 rows out to columns [col, col + 64)
// of each row whose bit is set in ok_rows, as whole lines.
__device__ __forceinline__ void stage_flush64(const GemmArgs& a, uint8_t* buf, int row0, int col, unsigned ok_rows) {
  const int lane = (int)(threadIdx.x & 31u);
  __syncwarp();
#pragma unroll
  for (int it = 0; it < 8; ++it) {
    const int r = it * 4 + (lane >> 3), u = lane & 7;
    if ((ok_rows >> r) & 1u)
      *reinterpret_cast<uint4*>(a.out + (size_t)(row0 + r) * a.ldo + col + u * 8) = *stage_unit(buf, r, u);
  }
  __syncwarp();
}

// Sixteen values as two staged 16-byte units of this lane's row.
__device__ __forceinline__ void stage16(uint8_t* buf, int u0, const float (&v)[16]) {
  const int lane = (int)(threadIdx.x & 31u);
#pragma unroll
  for (int g = 0; g < 2; ++g)
    *stage_unit(buf, lane, u0 + g) =
        make_uint4(pack_bf16x2(v[8 * g + 0], v[8 * g + 1]), pack_bf16x2(v[8 * g + 2], v[8 * g + 3]),
                   pack_bf16x2(v[8 * g + 4], v[8 * g + 5]), pack_bf16x2(v[8 * g + 6], v[8 * g + 7]));
}

// epi_qk_part through the warp's staging buffer, in two passes of 64
// channels: pass 1 holds the rotated channels 0..47 and their partners of
// band t (48..63); the partners of bands h and w (64..95) wait in registers
// as packed bf16 pairs while pass 1 is written, and join the normed
// channels 96..127 in pass 2.  Same arithmetic as epi_qk_part.
__device__ __forceinline__ void epi_qk_part_staged(const GemmArgs& a, uint32_t tpart, int m, bool valid, int h,
                                                   int part, const float (&pos)[3], uint8_t* buf) {
  const int lane = (int)(threadIdx.x & 31u);
  const int row0 = m - lane;
  const int cb = h * 384 + part * 128;       // output / weight column of channel 0
  const __nv_bfloat16* gain = part ? a.k_gain : a.q_gain;
  float ss = 0.f;
#pragma unroll 1
  for (int c = 0; c < 4; ++c) {
    uint32_t r[32];
    tmem_ld32(tpart + c * 32, r);
    tmem_ld_wait(r);
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const float v = bf16_round(__uint_as_float(r[j]) + bias_at(a.bias, cb + c * 32 + j));
      ss = __fmaf_rn(v, v, ss);
    }
  }
  const float inv = 1.0f / sqrtf(ss * (1.0f / 128.0f) + a.eps);
  const bool ok = valid && out_ok(a, a.out + (size_t)m * a.ldo + cb, 128, 6);
  const unsigned ok_rows = __ballot_sync(0xffffffffu, ok);
  uint32_t hold[16];                         // channels 64..95, packed pairs
#pragma unroll 1
  for (int band = 0; band < 3; ++band) {
    const float p = band == 0 ? pos[0] : (band == 1 ? pos[1] : pos[2]);
    uint32_t lo[16], hi[16];
    tmem_ld16(tpart + band * 16, lo);
    tmem_ld16(tpart + 48 + band * 16, hi);
    tmem_ld_wait(lo, hi);
    float o1[16], o2[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int j = band * 16 + i;
      float sn, cs;
      sincosf(p * a.omega[i], &sn, &cs);
      const float v1 = bf16_round(__uint_as_float(lo[i]) + bias_at(a.bias, cb + j));
      const float v2 = bf16_round(__uint_as_float(hi[i]) + bias_at(a.bias, cb + 48 + j));
      const float x1 = bf16_round(v1 * inv * __bfloat162float(gain[j]));
      const float x2 = bf16_round(v2 * inv * __bfloat162float(gain[48 + j]));
      o1[i] = __fmaf_rn(x1, cs, -(x2 * sn));
      o2[i] = __fmaf_rn(x2, cs, x1 * sn);
    }
    stage16(buf, 2 * band, o1);              // channels 16 band .. 16 band + 15
    if (band == 0) {
      stage16(buf, 6, o2);                   // channels 48..63
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint32_t w = pack_bf16x2(o2[2 * i], o2[2 * i + 1]);
        if (band == 1) hold[i] = w; else hold[8 + i] = w;
      }
    }
  }
  stage_flush64(a, buf, row0, cb, ok_rows);
#pragma unroll
  for (int g = 0; g < 4; ++g)                 // channels 64..95
    *stage_unit(buf, lane, g) = make_uint4(hold[4 * g], hold[4 * g + 1], hold[4 * g + 2], hold[4 * g + 3]);
  uint32_t r[32];
  tmem_ld32(tpart + 96, r);
  tmem_ld_wait(r);
  float v[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    const float x = bf16_round(__uint_as_float(r[j]) + bias_at(a.bias, cb + 96 + j));
    v[j] = x * inv * __bfloat162float(gain[96 + j]);
  }
#pragma unroll
  for (int g = 0; g < 4; ++g)                 // channels 96..127
    *stage_unit(buf, lane, 4 + g) =
        make_uint4(pack_bf16x2(v[8 * g + 0], v[8 * g + 1]), pack_bf16x2(v[8 * g + 2], v[8 * g + 3]),
                   pack_bf16x2(v[8 * g + 4], v[8 * g + 5]), pack_bf16x2(v[8 * g + 6], v[8 * g + 7]));
  stage_flush64(a, buf, row0, cb + 64, ok_rows);
}

// epi_v_head through the warp's staging buffer, two 64-column passes.
__device__ __forceinline__ void epi_v_head_staged(const GemmArgs& a, uint32_t tpart, int m, bool valid, int head,
                                                  uint8_t* buf) {
  const int lane = (int)(threadIdx.x & 31u);
  const int row0 = m - lane;
  const int cb = head * 384 + 256;
  const bool ok = valid && head < a.H && out_ok(a, a.out + (size_t)m * a.ldo + cb, 128, 9);
  const unsigned ok_rows = __ballot_sync(0xffffffffu, ok);
#pragma unroll 1
  for (int pass = 0; pass < 2; ++pass) {
#pragma unroll 1
    for (int cc = 0; cc < 2; ++cc) {
      const int c = 2 * pass + cc;
      uint32_t r[32];
      tmem_ld32(tpart + c * 32, r);
      tmem_ld_wait(r);
      float v[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]) + bias_at(a.bias, cb + c * 32 + j);
#pragma unroll
      for (int g = 0; g < 4; ++g)
        *stage_unit(buf, lane, cc * 4 + g) =
            make_uint4(pack_bf16x2(v[8 * g + 0], v[8 * g + 1]), pack_bf16x2(v[8 * g + 2], v[8 * g + 3]),
                       pack_bf16x2(v[8 * g + 4], v[8 * g + 5]), pack_bf16x2(v[8 * g + 6], v[8 * g + 7]));
    }
    stage_flush64(a, buf, row0, cb + 64 * pass, ok_rows);
  }
}

template <int BN>
__device__ __forceinline__ void epi_qkv(const GemmArgs& a, uint32_t tacc, int m, bool valid, int n_blk, int half,
                                        uint8_t* stage_buf) {
  float pos[3] = {0.f, 0.f, 0.f};
  if (valid) {
#pragma unroll
    for (int ax = 0; ax < 3; ++ax) {
      if (!in_bounds<int32_t>(a.pos, a.pos_elems, a.pos + (size_t)m * 3 + ax, 1, a.err, 18)) {
        valid = false;
        break;
      }
      const int p = a.pos[(size_t)m * 3 + ax];
      if ((unsigned)p >= (1u << 24)) {
        record_error(a.err, DEVERR_INDEX);
        valid = false;
      }
      pos[ax] = (float)p;
    }
  }
  if constexpr (BN == 256) {
    // q | k of head n_blk (one part per column half), or v of heads 2p, 2p+1
    if (n_blk < a.H) epi_qk_part_staged(a, tacc + half * 128, m, valid, n_blk, half, pos, stage_buf);
    else epi_v_head_staged(a, tacc + half * 128, m, valid, 2 * (n_blk - a.H) + half, stage_buf);
  } else if (half == 0) {
    // one 128-column part: its norm needs all of it in one warp
    const int head = n_blk / 3, part = n_blk % 3;
    if (part < 2) epi_qk_part(a, tacc, m, valid, head, part, pos);
    else epi_v_head(a, tacc, m, valid, head);
  }
}

// ---------------------------------------------------------------------------
// work items: whole tiles (unit, unit + num_units, ...) or, with stream-K, the
// tile pieces of this pair's run of k-blocks
// ---------------------------------------------------------------------------
struct WorkItem {
  int tile, k0, k1;
  bool owner;      // holds k-block 0 of the tile: finishes the tile
  bool sk;         // a stream-K piece (an owner then folds the partials of later runs)
};

// Stream-K runs: one lane of sk_lane pairs per 256-row tile (unit = m *
// sk_lane + j), all lanes walking the same column tiles and k-blocks at the
// same time (weights shared across the row tiles in L2); pair j of a lane
// takes k-blocks [j, j + 1) * sk_iters / sk_lane of the lane's num_n x num_k.
// In the tail form (sk_tail) pair j first runs its whole tiles j + i *
// sk_units of the first sk_dp tiles, then k-blocks [j, j + 1) * sk_iters /
// sk_units of the one lane over the tiles that follow.
__device__ __forceinline__ long long sk_start(const GemmArgs& a, int j) {
  return (long long)j * a.sk_iters / a.sk_lane;
}

__device__ __forceinline__ bool work_item(const GemmArgs& a, int unit, int num_units, int num_tiles, int i,
                                          WorkItem& w) {
  if (a.sk_units == 0) {
    w.tile = unit + i * num_units;
    w.k0 = 0;
    w.k1 = a.num_k;
    w.owner = true;
    w.sk = false;
    return w.tile < num_tiles;
  }
  int j, base;
  if (a.sk_tail) {
    // whole tiles first (as in a whole-tile launch), then this pair's run of
    // the one lane over the remaining tiles
    const int n_dp = a.sk_dp / num_units;
    if (i < n_dp) {
      w.tile = unit + i * num_units;
      w.k0 = 0;
      w.k1 = a.num_k;
      w.owner = true;
      w.sk = false;
      return true;
    }
    i -= n_dp;
    j = unit;
    base = a.sk_dp;
  } else {
    const int lane_m = unit / a.sk_lane;
    j = unit - lane_m * a.sk_lane;
    base = lane_m * a.num_n;         // m-major: (m, n) = (tile / num_n, tile % num_n)
  }
  const long long start = sk_start(a, j), end = sk_start(a, j + 1);
  const int n = (int)(start / a.num_k) + i;
  const long long tb = (long long)n * a.num_k;
  if (tb >= end) return false;
  w.tile = base + n;
  w.sk = true;
  w.k0 = i == 0 ? (int)(start - tb) : 0;
  w.k1 = end - tb < a.num_k ? (int)(end - tb) : a.num_k;
  w.owner = w.k0 == 0;
  return w.k0 < w.k1;
}

__device__ __forceinline__ float* sk_slot(const GemmArgs& a, int unit, uint32_t rank, int nchunks) {
  return a.sk_part + (size_t)(unit * 2 + (int)rank) * nchunks * (128 * 32);
}
// one flag per CTA, accumulator lane quadrant and column half (epilogue warp)
__device__ __forceinline__ uint32_t* sk_flag(const GemmArgs& a, int unit, uint32_t rank, int quad, int half) {
  return a.sk_flags + ((unit * 2 + (int)rank) * 4 + quad) * 2 + half;
}


// The i-th of the NCH/2 32-column accumulator chunks that the epilogue warps
// of column half `half` read: the first or second half of the tile, except
// for SwiGLU, where a half takes gate chunks and the value chunks paired with
// them (chunk c of the gate columns with chunk c of the value columns).
// Partial sums are stored and folded by the same warps that read them.
template <int EPI, int NCH>
__device__ __forceinline__ int sk_chunk(int half, int i) {
  if (EPI == EPI_SWIGLU)
    return i < NCH / 4 ? half * (NCH / 4) + i : NCH / 2 + half * (NCH / 4) + (i - NCH / 4);
  return half * (NCH / 2) + i;
}

// A piece that does not hold k-block 0: this warp's 32 accumulator rows
// (the 32-column chunks of its column half) to the pair's partial slot, then
// the warp's flag.
template <int EPI, int BN>
__device__ __forceinline__ void sk_store_partial(const GemmArgs& a, uint32_t tacc, int unit, uint32_t rank,
                                                 int quad, int half, int row, int lane) {
  constexpr int NCH = BN / 32;
  float* slot = sk_slot(a, unit, rank, NCH);
#pragma unroll 1
  for (int i = 0; i < NCH / 2; ++i) {
    const int c = sk_chunk<EPI, NCH>(half, i);
    uint32_t r[32];
    tmem_ld32(tacc + c * 32, r);
    tmem_ld_wait(r);
    // [chunk][16-byte group g][row]: one warp store covers 512 contiguous bytes
    uint4* d = reinterpret_cast<uint4*>(slot + (size_t)c * (128 * 32)) + row;
    if (in_bounds<float>(a.sk_part, a.sk_part_elems, slot + (size_t)c * (128 * 32), 128 * 32, a.err, 10)) {
#pragma unroll
      for (int g = 0; g < 8; ++g) d[g * 128] = make_uint4(r[4 * g], r[4 * g + 1], r[4 * g + 2], r[4 * g + 3]);
    }
  }
  __syncwarp();
  if (lane == 0) {
    __threadfence();
    st_release_u32(sk_flag(a, unit, rank, quad, half), a.sk_epoch);
  }
}

// The owner of tile `tile`: wait for the partials of the runs of its lane
// that start inside it (units unit+1, unit+2, ...; this warp's rows only) and
// add them, in that order, to the accumulator in TMEM.  Returns false
// (warp-uniform) when a wait gave up.
template <int EPI, int BN>
__device__ __forceinline__ bool sk_fold_partials(const GemmArgs& a, uint32_t tacc, int unit, uint32_t rank,
                                                 int quad, int half, int row, int lane, int tile,
                                                 const WaitCtl& abort_v) {
  constexpr int NCH = BN / 32;
  static_assert(NCH % 4 == 0, "each column half is folded two chunks at a time");
  const int j = unit % a.sk_lane;
  const long long lane_tile = a.sk_tail ? tile - a.sk_dp : tile % a.num_n;   // the tile's place in the lane
  const long long tile_end = (lane_tile + 1) * a.num_k;
  int j_end = j + 1;
  while (j_end < a.sk_lane && sk_start(a, j_end) < tile_end) ++j_end;
  const int q_end = unit + (j_end - j);
  if (q_end == unit + 1) return true;
  int ok = 1;
  if (lane == 0) {
    for (int q = unit + 1; q < q_end && ok; ++q) {
      const uint32_t* f = sk_flag(a, q, rank, quad, half);
      if (ld_acquire_u32(f) == a.sk_wait) continue;
      const uint64_t t0 = globaltimer();
      for (uint32_t i = 1;; ++i) {
        if (ld_acquire_u32(f) == a.sk_wait) break;
        if ((i & 31u) == 0 && wait_gives_up(abort_v, t0, kSiteStreamKFlag)) {
          ok = 0;
          break;
        }
      }
    }
  }
  ok = __shfl_sync(0xffffffffu, ok, 0);
  if (!ok) return false;
  // every lane acquires the flags it depends on before reading the partials
  for (int q = unit + 1; q < q_end; ++q) (void)ld_acquire_u32(sk_flag(a, q, rank, quad, half));
#pragma unroll 1
  for (int q = unit + 1; q < q_end; ++q) {
    const float* slot = sk_slot(a, q, rank, NCH);
    // (an out-of-range slot is reported; the bounds-checked build then reads
    // the first slot instead, so the warp's TMEM accesses stay uniform)
    if (!in_bounds<float>(a.sk_part, a.sk_part_elems, slot, (size_t)NCH * 128 * 32, a.err, 11)) slot = a.sk_part;
#pragma unroll 1
    for (int i = 0; i < NCH / 2; i += 2) {
      const int c = sk_chunk<EPI, NCH>(half, i);   // chunks c and c + 1 (pairs stay adjacent)
      float4 p[16];
      const float4* s0 = reinterpret_cast<const float4*>(slot + (size_t)c * (128 * 32)) + row;
      const float4* s1 = reinterpret_cast<const float4*>(slot + (size_t)(c + 1) * (128 * 32)) + row;
#pragma unroll
      for (int g = 0; g < 8; ++g) {
        p[g] = __ldcg(s0 + g * 128);
        p[8 + g] = __ldcg(s1 + g * 128);
      }
      uint32_t r0[32], r1[32];
      tmem_ld32(tacc + c * 32, r0);
      tmem_ld_wait(r0);
      tmem_ld32(tacc + (c + 1) * 32, r1);
      tmem_ld_wait(r1);
#pragma unroll
      for (int g = 0; g < 8; ++g) {
        r0[4 * g] = __float_as_uint(__uint_as_float(r0[4 * g]) + p[g].x);
        r0[4 * g + 1] = __float_as_uint(__uint_as_float(r0[4 * g + 1]) + p[g].y);
        r0[4 * g + 2] = __float_as_uint(__uint_as_float(r0[4 * g + 2]) + p[g].z);
        r0[4 * g + 3] = __float_as_uint(__uint_as_float(r0[4 * g + 3]) + p[g].w);
        r1[4 * g] = __float_as_uint(__uint_as_float(r1[4 * g]) + p[8 + g].x);
        r1[4 * g + 1] = __float_as_uint(__uint_as_float(r1[4 * g + 1]) + p[8 + g].y);
        r1[4 * g + 2] = __float_as_uint(__uint_as_float(r1[4 * g + 2]) + p[8 + g].z);
        r1[4 * g + 3] = __float_as_uint(__uint_as_float(r1[4 * g + 3]) + p[8 + g].w);
      }
      tmem_st32(tacc + c * 32, r0);
      tmem_st32(tacc + (c + 1) * 32, r1);
      tmem_st_wait();
    }
  }
  return true;
}

template <int EPI, int BN>
__device__ __forceinline__ void run_epilogue(const GemmArgs& a, uint32_t tacc, int m, int n_blk, int half,
                                             uint8_t* stage_buf) {
  const bool valid = m < a.M;
  if (EPI == EPI_PLAIN) epi_plain(a, tacc, m, valid, n_tile<EPI, BN>(a, n_blk), half);
  if (EPI == EPI_RESID) {
    if constexpr (gemm_staged_epi<EPI, BN>())
      epi_resid_staged(a, tacc, m, valid, n_tile<EPI, BN>(a, n_blk), half, n_blk, stage_buf);
    else
      epi_resid(a, tacc, m, valid, n_tile<EPI, BN>(a, n_blk), half, n_blk);
  }
  if constexpr (EPI == EPI_SWIGLU) {
    static_assert(gemm_staged_epi<EPI, BN>(), "SwiGLU tiles are 256 wide (128 gate + 128 value columns)");
    epi_swiglu_staged(a, tacc, m, valid, n_blk, half, stage_buf);
  }
  if (EPI == EPI_QKV) epi_qkv<BN>(a, tacc, m, valid, n_blk, half, stage_buf);
}

}  // namespace

template <int EPI, int BN>
__global__ void __launch_bounds__(GEMM_THREADS, 1)
    gemm_bf16_tc(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                 const GemmArgs args) {
  using C = GemmCfg<BN>;
  constexpr int STAGES = C::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * A_STAGE_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sB + STAGES * C::B_STAGE_BYTES);
  uint64_t* full = bars;                 // used in the even CTA: both CTAs' loads land on it
  uint64_t* empty = bars + STAGES;       // both CTAs: released by the pair's MMA commit
  uint64_t* acc_full = bars + 2 * STAGES;
  uint64_t* acc_empty = acc_full + 2;    // even CTA: 4 epilogue warps of each CTA
  uint64_t* drain = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);
  uint8_t* stage_base = reinterpret_cast<uint8_t*>(bars) + 256;   // epilogue staging (staged residual tiles)

  griddep_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();         // rank inside the CTA pair
  const bool leader = rank == 0;
  constexpr int CL = 2;
  const int unit = (int)(blockIdx.x / CL), num_units = (int)(gridDim.x / CL);
  const int num_tiles = args.num_m * args.num_n;
  const uint16_t pair_mask = 0x3;
  // tile `t` of this unit's walk -> (m_blk, n_blk) of this pair
  auto my_tile = [&](int t, int& m_blk, int& n_blk) {
    if (args.sk_units > 0 && !args.sk_tail) {
      m_blk = t / args.num_n;
      n_blk = t - m_blk * args.num_n;
      return;
    }
    tile_coords(t, args.num_m, args.num_n, m_blk, n_blk);
  };
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], 16);   // 8 epilogue warps of each CTA
    }
    mbar_init(drain, 1);
    *abort_flag = timeout_recorded(args.err) ? 1 : 0;   // sticky timeout of an earlier launch
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    // weights are never written: pull this CTA's half of the first tile into
    // L2 while the previous kernel on the stream may still be running
    WorkItem w0;
    if (work_item(args, unit, num_units, num_tiles, 0, w0)) {
      int m0, n0;
      my_tile(w0.tile, m0, n0);
      const int r0 = b_tile_row<EPI, BN>(args, n0, rank);
      for (int kb = w0.k0; kb < w0.k0 + C::STAGES + args.l2_pf && kb < w0.k1; ++kb)
        tma_prefetch_l2(&tmB, kb * BK, r0);
    }
  }
  if (warp == 1) tmem_alloc_pair(tmem_slot, 512);
  tc_fence_before();
  cluster_sync();          // barriers of both CTAs initialised, TMEM of both allocated
  tc_fence_after();
  griddep_wait();
  const uint32_t tmem_base = *tmem_slot;
  const WaitCtl abort_v{abort_flag, args.err, KID_GEMM};

  // a wait of an earlier launch ran out (sticky until h3_sync_check; read
  // in the prologue, beside the previous kernel): this launch skips its
  // work, before any copy or MMA is issued
  const bool skip = *abort_v.flag != 0;

  if (skip) {
  } else if (warp == 0) {
    // ---------------------------------------------------------- TMA producer (both CTAs)
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int last_phase[STAGES];
      for (int s = 0; s < STAGES; ++s) last_phase[s] = -1;
      bool ok = true;
      const uint32_t full0 = mapa_shared(smem_u32(full), 0);   // the even CTA's full[0]
      const uint32_t stage_tx = 2u * (uint32_t)(A_STAGE_BYTES + args.b_rows * BK * 2);   // both CTAs' boxes
      // stream-K: the activation rows are reused by every column tile of the
      // lane while each weight k-block is used once per row tile at about the
      // same time, so activations are kept in L2 ahead of the weight stream
      const uint64_t pol_a = l2_policy_evict_last(), pol_b = l2_policy_evict_first();
      WorkItem w;
      for (int i = 0; ok && work_item(args, unit, num_units, num_tiles, i, w); ++i) {
        int m_blk, n_blk;
        my_tile(w.tile, m_blk, n_blk);
        const int rb = b_tile_row<EPI, BN>(args, n_blk, rank);
        const int ra = m_blk * 2 * BM + (int)rank * BM;
        for (int kb = w.k0; kb < w.k1; ++kb) {
          if (!mbar_wait_cluster(&empty[stage], phase ^ 1u, abort_v)) { ok = false; break; }
          if (leader) mbar_arrive_expect_tx(&full[stage], stage_tx);
          const uint32_t fb = full0 + (uint32_t)stage * 8u;
          if (args.l2_hint) {
            tma_load_2d_pair_hint(sA + stage * A_STAGE_BYTES, &tmA, fb, kb * BK, ra, pol_a);
            tma_load_2d_pair_hint(sB + stage * C::B_STAGE_BYTES, &tmB, fb, kb * BK, rb, pol_b);
          } else {
            tma_load_2d_pair(sA + stage * A_STAGE_BYTES, &tmA, fb, kb * BK, ra);
            tma_load_2d_pair(sB + stage * C::B_STAGE_BYTES, &tmB, fb, kb * BK, rb);
          }
          last_phase[stage] = (int)phase;
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
          const int pk = kb + args.l2_pf;
          if (args.l2_pf > 0 && pk < w.k1) tma_prefetch_l2(&tmB, pk * BK, rb);
        }
      }
      if (ok) {
        // every stage handed out must come back (its release commit has landed)
        // before the CTA may exit
        for (int i = 0; i < STAGES && ok; ++i) {
          if (last_phase[stage] >= 0 && !mbar_wait_cluster(&empty[stage], phase ^ 1u, abort_v)) ok = false;
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
      } else if (leader) {  // let every load already issued land before the pair exits
        for (int s = 0; s < STAGES; ++s)
          if (last_phase[s] >= 0) drain_wait(&full[s], (uint32_t)last_phase[s]);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer (even CTA)
    if (lane == 0 && leader) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      int it = 0;
      WorkItem w;
      for (; ok && work_item(args, unit, num_units, num_tiles, it, w); ++it) {
        const int acc = it & 1;
        const uint32_t acc_phase = (uint32_t)(it >> 1) & 1u;
        if (!mbar_wait_cluster(&acc_empty[acc], acc_phase ^ 1u, abort_v)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
        int m_blk, n_blk;
        my_tile(w.tile, m_blk, n_blk);
        const uint32_t idesc = idesc_bf16(2 * BM, n_tile<EPI, BN>(args, n_blk).w);
        for (int kb = w.k0; kb < w.k1; ++kb) {
          if (!mbar_wait_cluster(&full[stage], phase, abort_v)) { ok = false; break; }
          tc_fence_after();
          const uint32_t a0 = smem_u32(sA + stage * A_STAGE_BYTES);
          const uint32_t b0 = smem_u32(sB + stage * C::B_STAGE_BYTES);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k) {
            mma_bf16_ss_pair(d_tmem, sdesc_kmajor(a0 + k * 32), sdesc_kmajor(b0 + k * 32), idesc,
                             (kb != w.k0 || k != 0) ? 1u : 0u);
          }
          mma_commit_pair(&empty[stage], pair_mask);
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        mma_commit_pair(&acc_full[acc], pair_mask);
      }
      if (!ok) {  // all MMAs issued so far must finish before TMEM is released
        mma_commit_pair(drain, (uint16_t)1u);
        drain_wait(drain, 0);
      }
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------- epilogue (both CTAs)
    const int q = warp & 3;              // TMEM lane quadrant
    const int half = (warp - 2) >> 2;    // column half: warps 2-5 first, 6-9 second
    const int row = q * 32 + lane;
    const uint32_t acc_empty0 = mapa_shared(smem_u32(acc_empty), 0);
    // fused norm: the tiles this warp owned (a stream-K run holds at most a
    // few whole tiles; a fourth and later one is not expected, see the host)
    constexpr int kMaxOwned = 4;
    int owned_m[kMaxOwned], owned_n[kMaxOwned], n_owned = 0;
    int it = 0;
    WorkItem w;
    for (; work_item(args, unit, num_units, num_tiles, it, w); ++it) {
      const int acc = it & 1;
      const uint32_t acc_phase = (uint32_t)(it >> 1) & 1u;
      if (!__all_sync(0xffffffffu, mbar_wait_cluster(&acc_full[acc], acc_phase, abort_v))) break;
      tc_fence_after();
      int m_blk, n_blk;
      my_tile(w.tile, m_blk, n_blk);
      const uint32_t tacc = tmem_addr(tmem_base, (uint32_t)(q * 32), (uint32_t)(acc * BN));
      bool done = true;
      if (!w.owner) {
        // stream-K piece without k-block 0: hand the partial to the owner
        // (stream-K launches use 256-column tiles only)
        if constexpr (BN == 256) sk_store_partial<EPI, BN>(args, tacc, unit, rank, q, half, row, lane);
      } else {
        if constexpr (BN == 256) {
          if (args.sk_units > 0 && w.sk) {
            if (EPI == EPI_RESID)
              epi_resid_prefetch(args, m_blk * 2 * BM + (int)rank * BM + row, n_tile<EPI, BN>(args, n_blk), half);
            done = sk_fold_partials<EPI, BN>(args, tacc, unit, rank, q, half, row, lane, w.tile, abort_v);
          }
        }
        if (done)
          run_epilogue<EPI, BN>(args, tacc, m_blk * 2 * BM + (int)rank * BM + row, n_blk, half,
                                stage_base + (warp - 2) * EPI_STAGE_WARP_BYTES);
        if (EPI == EPI_RESID && done && args.nrm_h) {
          // partial sums stored: count this warp for its row tile
          __syncwarp();
          if (lane == 0) {
            __threadfence();
            atomicAdd(args.nrm_cnt + m_blk, 1u);
          }
          if (n_owned < kMaxOwned) {
            owned_m[n_owned] = m_blk;
            owned_n[n_owned] = n_blk;
          }
          ++n_owned;
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(acc_empty0 + (uint32_t)acc * 8u);
      if (!done) break;
    }
    if (EPI == EPI_RESID && args.nrm_h) {
      if (n_owned > kMaxOwned) *abort_v.flag = 1;   // the host keeps runs shorter; never expected
      for (int i = 0; i < n_owned && i < kMaxOwned && !*abort_v.flag; ++i)
        if (!fused_norm(args, owned_m[i], owned_n[i], owned_m[i] * 2 * BM + (int)rank * BM + q * 32, half, lane,
                        abort_v))
          break;
    }
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();          // no CTA of the cluster still signals another's barriers or TMEM
  if (threadIdx.x == 0 && *abort_v.flag) record_error(args.err, DEVERR_TIMEOUT);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, 512);
  }
}

// ---------------------------------------------------------------------------
// host side: tile width choice and launch
// ---------------------------------------------------------------------------
int gemm_num_n(int epi, int bn, int N, int H, int F) {
  if (epi == EPI_SWIGLU) return F / 128;
  if (epi == EPI_QKV) return bn == 256 ? H + (H + 1) / 2 : 3 * H;
  return (N + bn - 1) / bn;
}

int gemm_b_box_rows(int epi, int bn) {
  (void)epi;
  return bn / 2;   // each CTA of a pair loads half of the tile's weight rows
}

int gemm_m_tiles(int M) { return (M + 2 * BM - 1) / (2 * BM); }

// Pick the tile width that minimises (waves x per-tile time) on this GPU.  A
// tile's time is its width over the per-SM efficiency measured for that width
// on GB300 (128-wide tiles feed the tensor core at about 65 % of the rate of
// 192- and 256-wide ones: each 128 x 128 x 16 MMA needs as many operand bytes
// per FLOP as the shared-memory port supplies).
// H3_GEMM_BN=256|192|128 in the environment forces one width where the
// epilogue supports it (tests sweep every width with it).
int gemm_choose_bn(int epi, int M, int N, int H, int F) {
  if (epi == EPI_SWIGLU) return 256;
  if (const char* env = getenv("H3_GEMM_BN")) {
    const int f = atoi(env);
    if (f == 256 || f == 128 || (f == 192 && epi != EPI_QKV)) return f;
  }
  const int slots = gemm_pair_slots();
  const int num_m = gemm_m_tiles(M);
  const int cands[3] = {256, 192, 128};
  int best = 256;
  long long best_cost = -1;
  for (int bn : cands) {
    if (epi == EPI_QKV && bn == 192) continue;
    const long long tiles = (long long)num_m * gemm_num_n(epi, bn, N, H, F);
    const long long waves = (tiles + slots - 1) / slots;
    const long long eff_pct = bn == 256 ? 100 : (bn == 192 ? 95 : 65);
    const long long cost = waves * bn * 100 / eff_pct;
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best = bn;
    }
  }
  return best;
}

// Balanced column widths: every 256-row tile gets `per_row` column tiles so
// that all of them are resident at once, widths nw1 and nw1 - 16 (multiples
// of 16).  Returns false when the uniform plan's wave model is at least as
// good.
static bool balance_columns(GemmPlan& p, int N, int num_m) {
  const int slots = gemm_pair_slots();
  const int per_row = slots / num_m;
  if (per_row < 1) return false;
  const int units = N / 16;
  const int u1 = (units + per_row - 1) / per_row;
  if (u1 < 4 || u1 > 16) return false;         // 64..256 columns
  const int u2 = u1 - 1;
  const int cnt1 = units - per_row * u2;       // cnt1 * u1 + (per_row - cnt1) * u2 == units
  const int cnt2 = per_row - cnt1;
  if (cnt1 < 1 || cnt1 > per_row) return false;
  // wave model of the uniform plan against one wave of the balanced one
  const long long u_tiles = (long long)num_m * p.num_n;
  const long long u_waves = (u_tiles + slots - 1) / slots;
  const long long u_cost = u_waves * p.bn * 100 / (p.bn == 256 ? 100 : (p.bn == 192 ? 95 : 65));
  const long long b_cost = (long long)(16 * u1) * 100 / 95;
  if (b_cost >= u_cost) return false;
  p.nw1 = 16 * u1;
  p.ncnt1 = cnt1;
  p.nw2 = cnt2 > 0 ? 16 * u2 : 0;
  p.num_n = per_row;
  p.bn = p.nw1 <= 128 ? 128 : (p.nw1 <= 192 ? 192 : 256);
  p.b_rows = p.nw1 / 2;
  return true;
}

GemmPlan gemm_plan(int epi, int M, int N, int H, int F) {
  GemmPlan p{};
  p.bn = gemm_choose_bn(epi, M, N, H, F);
  p.num_n = gemm_num_n(epi, p.bn, N, H, F);
  p.b_rows = gemm_b_box_rows(epi, p.bn);
  if ((epi != EPI_PLAIN && epi != EPI_RESID) || getenv("H3_GEMM_BN") || N % 16) return p;
  GemmPlan q = p;
  if (balance_columns(q, N, gemm_m_tiles(M))) return q;
  return p;
}

// Stream-K scratch for the largest launch: one slot of 256-column partial
// accumulators and 16 flags (CTA x lane quadrant x column half) per CTA pair
// that can be resident.
size_t gemm_sk_part_bytes() { return (size_t)gemm_pair_slots() * 2 * 128 * 256 * sizeof(float); }
size_t gemm_sk_flag_words() { return (size_t)gemm_pair_slots() * 16; }

// Whole 256-column tiles run in waves of one tile per resident pair (at most
// max_pairs when positive).  When the last wave would leave more than a
// tenth of the pairs idle (a few hundred rows: 505 rows x 5376 columns is 42
// tiles for 76 pairs; 256 rows x 21504 QKV columns 84), each
// 256-row tile gets a lane of floor(pairs / row tiles) pairs that share out
// its column tiles' k-blocks, provided that keeps nine tenths of the pairs
// busy and gives every pair at least 8 k-blocks.  Returns the pairs per lane.
int gemm_sk_lane(int M, int N, int K, int bn, int max_pairs) {
  const char* env = getenv("H3_GEMM_SK");
  if (env && env[0] == '0') return 0;
  const bool force = env && env[0] == '1';
  int slots = gemm_pair_slots();
  if (max_pairs > 0 && max_pairs < slots) slots = max_pairs;
  const int num_m = gemm_m_tiles(M);
  const long long num_n = (N + bn - 1) / bn;
  const long long lane_iters = num_n * (K / BK);
  if (num_m > slots) return 0;
  if (const char* u = getenv("H3_GEMM_SK_UNITS")) {
    // pairs in all: any lane width from 1 up to one k-block per pair (every
    // run nonempty: an owner waits for each later run that starts in its tile)
    long long lane = atoi(u) / num_m;
    if (lane > slots / num_m) lane = slots / num_m;
    if (lane > lane_iters) lane = lane_iters;
    if (lane >= 1) return (int)lane;
  }
  int lane = slots / num_m;
  if ((long long)lane * 8 > lane_iters) lane = (int)(lane_iters / 8);
  if (lane < 2) return 0;
  if (force) return lane;
  const long long tiles = (long long)num_m * num_n;
  const long long waves = (tiles + slots - 1) / slots;
  if (tiles * 10 >= waves * slots * 9) return 0;
  if ((long long)num_m * lane * 10 < (long long)slots * 9) return 0;
  return lane;
}

// Whole tiles, then stream-K over the tail: when whole 256-column tiles
// take more than one wave and the last wave would leave more than a tenth of
// the pairs idle (15,860 rows x 5376 columns: 1302 tiles, 17 waves of 76
// pairs and 10 tiles), the tiles of every full wave but the last run whole,
// and the rest (the last full wave and the partial one) are shared out over
// all pairs as one stream-K lane, each pair's run following its whole tiles.
// Returns the number of whole tiles (a multiple of *units), or -1 when the
// split does not apply (it needs at least 8 k-blocks per pair in the tail).
// H3_GEMM_SK=0 turns it off; H3_GEMM_SK_TAIL=n forces it with n pairs (tests).
int gemm_sk_tail(int M, int N, int K, int bn, int* units) {
  const char* env = getenv("H3_GEMM_SK");
  if (env && env[0] == '0') return -1;
  const long long tiles = (long long)gemm_m_tiles(M) * ((N + bn - 1) / bn);
  const long long num_k = K / BK;
  int slots = gemm_pair_slots();
  const char* forced = getenv("H3_GEMM_SK_TAIL");
  if (forced) {
    const int f = atoi(forced);
    if (f < 1 || f > slots) return -1;
    slots = f;
  } else {
    if (slots < 1 || tiles <= slots) return -1;
    const long long rem = tiles % slots;
    if (rem == 0 || rem * 10 >= (long long)slots * 9) return -1;
  }
  const long long full = tiles / slots;
  const long long dp = full > 0 ? (full - 1) * slots : 0;
  if ((tiles - dp) * num_k < (forced ? 1LL : 8LL) * slots) return -1;
  *units = slots;
  return (int)dp;
}

// CTA pairs that can be resident at once.
int gemm_pair_slots() {
  static int slots[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = 0;
  if (!slots[dev]) {
    // every instance holds one CTA per SM; the largest shared-memory footprint bounds them all
    constexpr int smem = GemmCfg<192>::SMEM > GemmCfg<256>::SMEM ? GemmCfg<192>::SMEM : GemmCfg<256>::SMEM;
    int n = 0;
    if (cudaFuncSetAttribute(gemm_bf16_tc<EPI_PLAIN, 192>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) ==
        cudaSuccess) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(2 * 1024);
      cfg.blockDim = dim3(GEMM_THREADS);
      cfg.dynamicSmemBytes = smem;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = 2;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      if (cudaOccupancyMaxActiveClusters(&n, gemm_bf16_tc<EPI_PLAIN, 192>, &cfg) != cudaSuccess) n = 0;
    }
    cudaGetLastError();
    slots[dev] = n > 0 ? n : (num_sms() / 2 > 0 ? num_sms() / 2 : 1);
  }
  return slots[dev];
}

template <int EPI, int BN>
static cudaError_t launch_one(const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmArgs& a, int grid,
                              cudaStream_t stream) {
  constexpr int smem = gemm_smem<EPI, BN>();
  static_assert(tmem_footprint_exclusive(smem), "a GEMM CTA must hold its SM's TMEM alone");
  if (!tmem_exclusive(smem)) return cudaErrorNotSupported;
  cudaError_t e = cudaFuncSetAttribute(gemm_bf16_tc<EPI, BN>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  return launch_kernel_cluster(gemm_bf16_tc<EPI, BN>, dim3(grid), dim3(GEMM_THREADS), smem, stream, 2, tmA, tmB, a);
}

cudaError_t launch_gemm(int epi, int bn, const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmArgs& args,
                        cudaStream_t stream) {
  // Weight L2 prefetch distance in k-blocks.  Measured on GB300: with up to
  // 16 row tiles (4096 rows) the TMA ring alone is faster by 1-5 %; at
  // 15860 rows prefetching two rings ahead is faster by up to 7 %.
  // H3_GEMM_L2PF=<k-blocks> overrides it.
  const int stages = bn == 256 ? GemmCfg<256>::STAGES : (bn == 192 ? GemmCfg<192>::STAGES : GemmCfg<128>::STAGES);
  GemmArgs a = args;
  // buffer extents implied by the arguments (checked by the bounds-checked build)
  a.out_elems = (size_t)a.M * a.ldo;
  a.resid_elems = a.resid ? (size_t)a.M * a.ldr : 0;
  a.table_elems = a.table ? (size_t)3 * a.T * 6 * a.D : 0;
  a.pos_elems = a.pos ? (size_t)3 * a.M : 0;
  a.sk_part_elems = gemm_sk_part_bytes() / sizeof(float);
  const char* pf = getenv("H3_GEMM_L2PF");
  const int pf_default = a.num_m <= 16 ? 0 : 2 * stages;
  a.l2_pf = pf ? atoi(pf) : pf_default;
  if (a.l2_pf < 0 || a.l2_pf > 256) a.l2_pf = pf_default;
  const int tiles = a.num_m * a.num_n;
  const int slots = gemm_pair_slots();
  int pairs = tiles < slots ? tiles : slots;
  if (a.max_ctas > 0 && pairs > a.max_ctas / 2) pairs = a.max_ctas / 2 > 0 ? a.max_ctas / 2 : 1;
  if (a.sk_units > 0) {
    // every pair of a stream-K launch must be resident: an owner waits for
    // the partials of later pairs
    if (bn != 256 || a.sk_units > slots) return cudaErrorInvalidValue;
    pairs = a.sk_units;
  }
  const int grid = 2 * pairs;
  const char* names[4] = {"plain", "qkv_qknorm_rope", "gated_residual", "swiglu"};
  cudaError_t e = cudaErrorInvalidValue;
#define H3_GEMM_CASE(E, B)                      \
  case E * 1000 + B:                            \
    e = launch_one<E, B>(tmA, tmB, a, grid, stream); \
    break;
  switch (epi * 1000 + bn) {
    H3_GEMM_CASE(EPI_PLAIN, 256)
    H3_GEMM_CASE(EPI_PLAIN, 192)
    H3_GEMM_CASE(EPI_PLAIN, 128)
    H3_GEMM_CASE(EPI_RESID, 256)
    H3_GEMM_CASE(EPI_RESID, 192)
    H3_GEMM_CASE(EPI_RESID, 128)
    H3_GEMM_CASE(EPI_QKV, 256)
    H3_GEMM_CASE(EPI_QKV, 128)
    H3_GEMM_CASE(EPI_SWIGLU, 256)
    default: return cudaErrorInvalidValue;
  }
#undef H3_GEMM_CASE
  if (e != cudaSuccess) return e;
  set_kernel_info("gemm_bf16_tc<%s,%d> tcgen05.mma.cta_group::2.kind::f16 pair-tile=%dx%dx%d stages=%d acc=f32 "
                  "tmem=2x%d grid=%d (pairs=%d of %d) tiles=%dx%d k_blocks=%d l2_prefetch=%d stream-k=%d "
                  "sk-whole-tiles=%d l2-hint=%d n-widths=%s%d,%d,%d",
                  names[epi], bn, 2 * BM, bn, BK, stages, bn, grid, pairs, slots, a.num_m, a.num_n, a.num_k,
                  a.l2_pf, a.sk_units, a.sk_tail ? a.sk_dp : -1, a.l2_hint, a.nw1 ? "balanced:" : "uniform:",
                  a.nw1 ? a.nw1 : bn, a.ncnt1, a.nw2);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// AdaLN table
// ---------------------------------------------------------------------------
namespace {
constexpr int AD_KPS = 2;       // 64-column boxes per stage (256 contiguous bytes of each weight row)
constexpr int AD_STAGES = 4;
constexpr int AD_STAGE_BYTES = AD_KPS * A_STAGE_BYTES;
constexpr int AD_BN = 16;
constexpr int AD_THREADS = 192;
constexpr int AD_U_MAX_KB = kMaxCondDim / 64;  // 64-column blocks of u held in shared memory
static_assert(AD_U_MAX_KB * 64 == kMaxCondDim, "the widest conditioning is a whole number of 64-column blocks");
constexpr int AD_SMEM = 1024 + AD_U_MAX_KB * 2048 + AD_STAGES * AD_STAGE_BYTES + 256;
}  // namespace

// u[t][k] = bf16(SiLU(t_cond[t][k])) in fp32 for t < T, zero for T <= t < 16;
// also zeroes n_zero words (the stream-K flags of the block call it starts).
__global__ void __launch_bounds__(256) silu_rows_kernel(const float* __restrict__ t_cond, int T, int C,
                                                        __nv_bfloat16* __restrict__ u, uint32_t* zero_words,
                                                        int n_zero) {
  griddep_launch_dependents();
  griddep_wait();
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n_zero; i += gridDim.x * blockDim.x) zero_words[i] = 0u;
  const int n = AD_BN * C;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
    const int t = i / C;
    float v = 0.0f;
    if (t < T) {
      const float x = t_cond[i];
      v = x / (1.0f + expf(-x));
    }
    u[i] = __float2bfloat16_rn(v);
  }
}

// NM = 1: one block's table (the weight map and bias in maps[0]); NM =
// kAdalnBatch: the tables of args.n_blocks blocks, tile t of the launch being
// tile t % (tiles per block) of block t / (tiles per block).
template <int NM>
__global__ void __launch_bounds__(AD_THREADS, 1)
    adaln_table_kernel(const __grid_constant__ AdalnMaps<NM> maps, const __grid_constant__ CUtensorMap tmU,
                       const AdalnArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  const int nkb = args.C / BK;                 // 64-column blocks of K
  const int nst = (nkb + AD_KPS - 1) / AD_KPS; // stages per tile
  uint8_t* sU = smem;                          // nkb blocks of 16 rows x 128 B
  uint8_t* sA = smem + nkb * 2048;             // 1024-aligned (2048 multiple)
  uint64_t* bars = reinterpret_cast<uint64_t*>(sA + AD_STAGES * AD_STAGE_BYTES);
  uint64_t* full = bars;
  uint64_t* empty = bars + AD_STAGES;
  uint64_t* acc_full = bars + 2 * AD_STAGES;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* u_full = acc_empty + 2;
  uint64_t* drain = u_full + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);

  griddep_launch_dependents();
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
    mbar_init(u_full, 1);
    mbar_init(drain, 1);
    *abort_flag = timeout_recorded(args.err) ? 1 : 0;   // sticky timeout of an earlier launch
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, 32);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // tiles of chunks [chunk_lo, chunk_hi) of every modality, of every block
  const int tiles_per_mod = (args.chunk_hi - args.chunk_lo) * args.D / BM;
  const int tiles_per_blk = 3 * tiles_per_mod;
  const int num_tiles = tiles_per_blk * (NM == 1 ? 1 : args.n_blocks);
  auto tile_blk = [&](int tile) { return NM == 1 ? 0 : tile / tiles_per_blk; };
  auto tile_row = [&](int tile) {
    const int lt = NM == 1 ? tile : tile % tiles_per_blk;
    const int m = lt / tiles_per_mod;
    return m * 6 * args.D + args.chunk_lo * args.D + (lt - m * tiles_per_mod) * BM;
  };
  const WaitCtl abort_v{abort_flag, args.err, KID_ADALN};
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmU);
    // weights are never written: pull the first tile's into L2 while the
    // previous kernel (the SiLU rows) may still be running
    if ((int)blockIdx.x < num_tiles) {
      const CUtensorMap* tw = &maps.w[tile_blk(blockIdx.x)];
      tma_prefetch_desc(tw);
      const int row0 = tile_row(blockIdx.x);
      for (int kb = 0; kb < (AD_STAGES + args.l2_pf) * AD_KPS && kb < nkb; ++kb)
        tma_prefetch_l2(tw, kb * BK, row0);
    }
  }
  griddep_wait();

  // a wait of an earlier launch ran out (sticky until h3_sync_check; read
  // in the prologue, beside the previous kernel): this launch skips its
  // work, before any copy or MMA is issued
  const bool skip = *abort_v.flag != 0;

  if (skip) {
  } else if (warp == 0) {
    if (lane == 0) {
      // the resident N = 16 operand, one 2 KB box per 64 columns of K
      mbar_arrive_expect_tx(u_full, (uint32_t)nkb * 2048u);
      for (int kb = 0; kb < nkb; ++kb) tma_load_2d(sU + kb * 2048, &tmU, u_full, kb * BK, 0);
      int stage = 0;
      uint32_t phase = 0;
      int last_phase[AD_STAGES];
      for (int s = 0; s < AD_STAGES; ++s) last_phase[s] = -1;
      bool ok = true;
      for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
        const int row0 = tile_row(tile);
        const CUtensorMap* tw = &maps.w[tile_blk(tile)];
        for (int kb = 0; kb < args.l2_pf * AD_KPS && kb < nkb; ++kb) tma_prefetch_l2(tw, kb * BK, row0);
        for (int st = 0; st < nst; ++st) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, abort_v)) { ok = false; break; }
          const int k0 = st * AD_KPS;
          const int nb = nkb - k0 < AD_KPS ? nkb - k0 : AD_KPS;
          mbar_arrive_expect_tx(&full[stage], (uint32_t)(nb * A_STAGE_BYTES));
          for (int b = 0; b < nb; ++b)
            tma_load_2d(sA + stage * AD_STAGE_BYTES + b * A_STAGE_BYTES, tw, &full[stage], (k0 + b) * BK,
                        row0);
          last_phase[stage] = (int)phase;
          if (++stage == AD_STAGES) { stage = 0; phase ^= 1u; }
          for (int b = 0; b < AD_KPS && args.l2_pf > 0; ++b) {
            const int pk = (st + args.l2_pf) * AD_KPS + b;
            if (pk < nkb) tma_prefetch_l2(tw, pk * BK, row0);
          }
        }
      }
      if (!ok) {
        drain_wait(u_full, 0);
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
      bool ok = mbar_wait(u_full, 0, abort_v);
      int it = 0;
      const uint32_t u0 = smem_u32(sU);
      for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x, ++it) {
        const int acc = it & 1;
        const uint32_t acc_phase = (uint32_t)(it >> 1) & 1u;
        if (!mbar_wait(&acc_empty[acc], acc_phase ^ 1u, abort_v)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * AD_BN);
        for (int st = 0; st < nst; ++st) {
          if (!mbar_wait(&full[stage], phase, abort_v)) { ok = false; break; }
          tc_fence_after();
          const int k0 = st * AD_KPS;
          const int nb = nkb - k0 < AD_KPS ? nkb - k0 : AD_KPS;
          for (int b = 0; b < nb; ++b) {
            const uint32_t a0 = smem_u32(sA + stage * AD_STAGE_BYTES + b * A_STAGE_BYTES);
            const uint32_t b0 = u0 + (uint32_t)(k0 + b) * 2048u;
#pragma unroll
            for (int k = 0; k < BK / 16; ++k) {
              mma_bf16_ss(d_tmem, sdesc_kmajor(a0 + k * 32), sdesc_kmajor(b0 + k * 32), idesc,
                          ((k0 + b) | k) != 0 ? 1u : 0u);
            }
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
      const int n = tile_row(tile) + row;
      const int blk = tile_blk(tile);
      const float b = bias_at(maps.bias[blk], n);
      __nv_bfloat16* out = args.out + (size_t)blk * args.out_block_stride;
#pragma unroll
      for (int t = 0; t < AD_BN; ++t) {
        if (t < args.T) out[(size_t)t * args.NW + n] = __float2bfloat16_rn(__uint_as_float(r[t]) + b);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0 && *abort_v.flag) record_error(args.err, DEVERR_TIMEOUT);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 32);
  }
}

cudaError_t launch_silu_rows(const float* t_cond, int T, int C, __nv_bfloat16* u, uint32_t* zero_words,
                             int n_zero_words, cudaStream_t stream) {
  const int n = AD_BN * C;
  const int blocks = (n + 255) / 256 < 1024 ? (n + 255) / 256 : 1024;
  return launch_kernel(silu_rows_kernel, dim3(blocks), dim3(256), 0, stream, t_cond, T, C, u, zero_words,
                       zero_words ? n_zero_words : 0);
}

static int adaln_l2_prefetch() {
  // Prefetching the weight stream into L2 ahead of the TMA loads measured
  // slower on GB300 (6.2 against 6.6 TB/s over the full table, 35 against
  // 31 us for chunks 0-1 at D = 5376): the ring alone keeps HBM busy.  Only
  // the first tile's stages are prefetched, before the dependency wait.
  // H3_ADALN_L2PF=<stages> turns the running prefetch on.
  const char* pf = getenv("H3_ADALN_L2PF");
  const int v = pf ? atoi(pf) : 0;
  return v < 0 || v > 64 ? 0 : v;
}

template <int NM>
static cudaError_t launch_adaln_kernel(const AdalnMaps<NM>& maps, const CUtensorMap& tmU, const AdalnArgs& a,
                                       int grid, int cluster, cudaStream_t stream) {
  static_assert(tmem_footprint_exclusive(AD_SMEM), "an AdaLN-table CTA must hold its SM's TMEM alone");
  if (!tmem_exclusive(AD_SMEM)) return cudaErrorNotSupported;
  cudaError_t e =
      cudaFuncSetAttribute(adaln_table_kernel<NM>, cudaFuncAttributeMaxDynamicSharedMemorySize, AD_SMEM);
  if (e != cudaSuccess) return e;
  return launch_kernel_cluster(adaln_table_kernel<NM>, dim3(grid), dim3(AD_THREADS), AD_SMEM, stream, cluster, maps,
                               tmU, a);
}

cudaError_t launch_adaln_table(const CUtensorMap& tmW, const CUtensorMap& tmU, const AdalnArgs& a,
                               cudaStream_t stream) {
  const int tiles = 3 * (a.chunk_hi - a.chunk_lo) * a.D / BM;
  int grid = tiles < num_sms() ? tiles : num_sms();
  // Sharing the GPU with a GEMM (max_ctas > 0): launch in clusters of two so
  // that the CTAs take whole SM pairs and leave whole pairs to the GEMM's CTA
  // pairs (single CTAs spread one per pair would strand the other SM).
  int cluster = 1;
  if (a.max_ctas > 0) {
    if (grid > a.max_ctas) grid = a.max_ctas;
    if (grid >= 2) {
      grid &= ~1;
      cluster = 2;
    }
  }
  AdalnArgs a2 = a;
  a2.l2_pf = adaln_l2_prefetch();
  a2.n_blocks = 1;
  AdalnMaps<1> maps;
  maps.w[0] = tmW;
  maps.bias[0] = a.bias;
  cudaError_t e = launch_adaln_kernel(maps, tmU, a2, grid, cluster, stream);
  if (e != cudaSuccess) return e;
  set_kernel_info("adaln_table_kernel tcgen05.mma.cta_group::1.kind::f16 tile=%dx%dx%d stages=%dx%d acc=f32 "
                  "tmem=2x%d grid=%d cluster=%d tiles=%d chunks=[%d,%d) k_blocks=%d l2_prefetch=%d stages",
                  BM, AD_BN, BK, AD_STAGES, AD_KPS, AD_BN, grid, cluster, tiles, a.chunk_lo, a.chunk_hi, a.C / BK,
                  a2.l2_pf);
  return cudaGetLastError();
}

cudaError_t launch_adaln_tables_batched(const AdalnBatchMaps& maps, const CUtensorMap& tmU, const AdalnArgs& a,
                                        cudaStream_t stream) {
  if (a.n_blocks < 1 || a.n_blocks > kAdalnBatch) return cudaErrorInvalidValue;
  const long long tiles = 3LL * (a.chunk_hi - a.chunk_lo) * a.D / BM * a.n_blocks;
  const int grid = tiles < num_sms() ? (int)tiles : num_sms();
  AdalnArgs a2 = a;
  a2.l2_pf = adaln_l2_prefetch();
  cudaError_t e = launch_adaln_kernel(maps, tmU, a2, grid, 1, stream);
  if (e != cudaSuccess) return e;
  set_kernel_info("adaln_table_kernel<batched> tcgen05.mma.cta_group::1.kind::f16 tile=%dx%dx%d stages=%dx%d "
                  "acc=f32 tmem=2x%d grid=%d blocks=%d tiles=%lld k_blocks=%d", BM, AD_BN, BK, AD_STAGES, AD_KPS,
                  AD_BN, grid, a.n_blocks, tiles, a.C / BK);
  return cudaGetLastError();
}

}  // namespace h3
