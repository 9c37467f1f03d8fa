// Host-side declarations shared by the translation units of libh3: kernel
// argument blocks, launchers and the tensor-map helper.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace h3 {

// ---------------------------------------------------------------------------
// tensor maps (cuTensorMapEncodeTiled through the runtime's driver entry point)
// ---------------------------------------------------------------------------
// 2-D bf16 tensor [rows][cols] with row stride `ld` elements, box
// [box_rows][64] (64 bf16 = 128 bytes), 128-byte swizzle, zero OOB fill.
bool make_tmap_2d(CUtensorMap* tm, const void* base, uint64_t rows, uint64_t cols, uint64_t ld,
                  uint32_t box_rows);
// 3-D bf16 tensor (channel c < 128, head h < H, row i < S) at
// base + i*row_stride + h*head_stride + c, box (64, 1, box_rows).
bool make_tmap_qkv(CUtensorMap* tm, const void* base, uint64_t n_rows, uint64_t n_heads,
                   uint64_t row_stride, uint64_t head_stride, uint32_t box_rows);

int num_sms();

// Launch with programmatic stream serialization (the kernel may start while
// the previous kernel on the stream finishes; it synchronises with
// griddepcontrol.wait).  H3_NO_PDL=1 in the environment launches without it.
bool pdl_enabled();
// cluster_x > 1 launches clusters of cluster_x CTAs along x.  early = false
// launches in plain stream order (griddepcontrol.wait then returns at once;
// the kernel's own griddepcontrol.launch_dependents still lets the next
// kernel start early).
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel_ex(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                             int cluster_x, bool early, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  int n = 0;
  if (early && pdl_enabled()) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  if (cluster_x > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = (unsigned)cluster_x;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel_cluster(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                                  int cluster_x, Args&&... args) {
  return launch_kernel_ex(kernel, grid, block, smem, stream, cluster_x, true, static_cast<Args&&>(args)...);
}
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                          Args&&... args) {
  return launch_kernel_ex(kernel, grid, block, smem, stream, 1, true, static_cast<Args&&>(args)...);
}
// Device address of the error words of the current device: [0] the error
// bits (DEVERR_*), [1] the site of the first timed-out wait (kernel id in the
// top byte, the barrier's shared-memory offset / 8 or kSiteStreamKFlag below).
uint32_t* device_error_word();

// ---------------------------------------------------------------------------
// TMEM exclusivity.  Every kernel that allocates tensor memory (the GEMM, both
// attention kernels, the AdaLN table) allocates before griddepcontrol.wait,
// so that the allocation overlaps the previous kernel's tail, and the
// allocation blocks until the columns are free.  That is safe only while no
// two such CTAs can be resident on one SM at the same time: a dependent CTA
// holding TMEM on an SM where a primary CTA has started but not yet allocated
// would wait for that primary grid forever.  The kernels keep it by their
// shared-memory footprint: each takes more than half of an SM's shared
// memory, so a second CTA of any of them cannot be placed beside it.  The
// static checks below pin the footprints against the sm_100-family figure
// (228 KB per SM, 1 KB reserved per CTA); tmem_exclusive() repeats the check
// against the figures the device reports, once per device, and the launchers
// refuse to launch when it fails.
// ---------------------------------------------------------------------------
constexpr int kSmemPerSm = 233472;
constexpr int kSmemReservedPerCta = 1024;
constexpr bool tmem_footprint_exclusive(int dyn_smem) {
  return 2 * (dyn_smem + kSmemReservedPerCta) > kSmemPerSm;
}
bool tmem_exclusive(int dyn_smem);
void set_kernel_info(const char* fmt, ...);

// ---------------------------------------------------------------------------
// GEMM (tcgen05 CTA pairs, 256 x BN x 64 tiles, persistent, warp-specialised)
// ---------------------------------------------------------------------------
enum GemmEpilogue : int {
  EPI_PLAIN = 0,   // y = bf16(acc + b)
  EPI_QKV = 1,     // per-head Q/K RMSNorm + MM-RoPE on q|k tiles, plain v tiles
  EPI_RESID = 2,   // y = bf16(x + gate[r] * bf16(acc + b))
  EPI_SWIGLU = 3,  // a = bf16(SiLU(bf16(acc_g + b_g)) * bf16(acc_u + b_u))
};

struct GemmArgs {
  int M;                 // rows of the activation operand (packed rows S)
  int K;                 // reduction length (multiple of 64)
  int num_m, num_n, num_k;
  __nv_bfloat16* out;    // output, row stride ldo elements
  int ldo;
  const __nv_bfloat16* bias;  // nullable; indexed by the weight row
  int n_valid;           // PLAIN / RESID: number of output columns
  // RESID: gate chunk of the AdaLN table and the residual input
  const __nv_bfloat16* resid;
  int ldr;
  const __nv_bfloat16* table;  // [3T][6][D]
  int D, chunk, T;
  const int32_t* tag;
  const int32_t* tidx;
  // SWIGLU
  int F;
  // QKV
  int H;
  const __nv_bfloat16* q_gain;
  const __nv_bfloat16* k_gain;
  const int32_t* pos;
  float eps;
  float omega[16];
  int max_ctas;          // 0: one CTA per SM; otherwise at most this many
  // column tiling (see GemmPlan): b_rows weight rows per CTA and k-block;
  // nw1 = 0 for uniform tiles of BN columns
  int b_rows;
  int nw1, ncnt1, nw2;
  int l2_pf;             // k-blocks of weight L2 prefetch ahead of the loads (0: none); set by launch_gemm
  int l2_hint;           // 1: activation tiles loaded evict-last, weight tiles evict-first (set with stream-K)
  // stream-K (sk_units > 0, pairs only): each 256-row tile has a lane of
  // sk_lane CTA pairs; the lane's num_n column tiles x num_k k-blocks,
  // column-tile-major, are cut into sk_lane equal runs.  A run that starts
  // inside a tile writes that tile's partial accumulator to sk_part and sets
  // its flags to sk_epoch; the pair whose run holds the tile's first k-block
  // adds the partials (in k order) and runs the epilogue.
  // With sk_tail = 1 there is one lane instead, over all sk_units pairs:
  // the first sk_dp tiles (a multiple of sk_units) run whole, tile u + i *
  // sk_units on pair u as in a whole-tile launch, and the k-blocks of tiles
  // [sk_dp, num_m * num_n) (in the whole-tile launch order) are cut into
  // sk_units equal runs that follow them.
  int sk_units;          // num_m * sk_lane, or the pairs of the one lane (sk_tail)
  int sk_lane;           // pairs per 256-row tile (sk_tail: sk_units)
  long long sk_iters;    // the k-blocks of one lane: num_n * num_k (sk_tail: the tail tiles' k-blocks)
  int sk_tail;           // 1: whole tiles first, then one stream-K lane over the remaining tiles
  int sk_dp;             // sk_tail: the tiles that run whole
  float* sk_part;        // [sk_units][2 CTAs][BN/32 chunks][8 groups][128 rows][4] fp32
  uint32_t* sk_flags;    // [sk_units][2 CTAs][4 row quadrants][2 column halves], zero before first use
  uint32_t sk_epoch;     // nonzero, distinct for every launch between two zeroings
  uint32_t sk_wait;      // the flag value owners wait for: sk_epoch (see gemm_set_sk for the test hook)
  // RESID with the following RMSNorm + modulation fused (stream-K launches,
  // where every pair is resident): each owner warp also stores, per row, the
  // sum of squares of the bf16 outputs of its column half into nrm_part and
  // counts itself in nrm_cnt[row tile]; after all its tiles, it waits until
  // the row tile's count reaches nrm_target and writes
  //   nrm_h = bf16((out * inv) * gain * (1 + table[scale]) + table[shift]),
  //   inv = 1 / sqrt(sum of the row's partials in column order / D + eps),
  // for the columns it owns.
  __nv_bfloat16* nrm_h;           // [M][D], null when not fused
  const __nv_bfloat16* nrm_gain;  // [D]
  int nrm_shift, nrm_scale;       // table chunks of the modulation
  float* nrm_part;                // [num_m * 256][2 * num_n]
  uint32_t* nrm_cnt;              // [num_m], zeroed with the stream-K flags
  uint32_t nrm_target;            // 16 * num_n arrivals per fused launch since that zeroing
  // extents (elements) for the bounds-checked build: out, resid, the AdaLN
  // table, positions and the stream-K partial area
  size_t out_elems, resid_elems, table_elems, pos_elems, sk_part_elems;
  uint32_t* err;
};

// Stream-K scratch of one GEMM launch inside a block call: partial
// accumulators and flags (see GemmArgs), the flags zeroed by the first kernel
// of the call.  epoch counts the launches that used them since.
struct SkScratch {
  float* part;
  uint32_t* flags;
  uint32_t epoch;
  float* nrm_part;        // fused-norm partial sums of squares (see GemmArgs)
  uint32_t* nrm_cnt;      // fused-norm arrival counters, zeroed with the flags
  uint32_t nrm_launches;  // fused launches since the zeroing
};
size_t gemm_sk_part_bytes();    // partial area for the largest stream-K launch on this GPU
size_t gemm_sk_flag_words();    // flags for the largest stream-K launch on this GPU
// CTA pairs per 256-row tile of a stream-K launch of this GEMM (on at most
// max_pairs pairs when positive), 0 when whole tiles per pair are at least
// as good.  H3_GEMM_SK=0 turns stream-K off, =1
// forces it on whenever it is possible; H3_GEMM_SK_UNITS=<n> forces it with
// n / row tiles pairs per row tile (at most one k-block per pair).
int gemm_sk_lane(int M, int N, int K, int bn, int max_pairs);
int gemm_sk_tail(int M, int N, int K, int bn, int* units);

// Column tiling of one GEMM launch.  Uniform: num_n tiles of bn columns.
// Balanced (plain and residual epilogues, when one wave of uniform tiles
// would leave CTA pairs idle): the N columns of each 256-row tile are split
// into ncnt1 tiles of nw1 columns followed by tiles of nw2 = nw1 - 16, as many
// as the resident pairs allow for all row tiles at once; bn is then the
// compiled width that holds nw1.  b_rows: weight rows one CTA loads per
// k-block (the B box of the tensor map).
struct GemmPlan {
  int bn, num_n, b_rows;
  int nw1, ncnt1, nw2;
};
GemmPlan gemm_plan(int epi, int M, int N, int H, int F);
// Tile width (256, 192 or 128 columns) for uniform tiles of a GEMM of M rows;
// the number of N tiles and the row count of one B box at that width.
int gemm_choose_bn(int epi, int M, int N, int H, int F);
int gemm_num_n(int epi, int bn, int N, int H, int F);
int gemm_b_box_rows(int epi, int bn);
int gemm_m_tiles(int M);        // 256-row tiles (one per CTA pair)
int gemm_pair_slots();          // CTA pairs that can be resident at once on this GPU
cudaError_t launch_gemm(int epi, int bn, const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmArgs& a,
                        cudaStream_t stream);

// AdaLN table: u = bf16(SiLU(t_cond)) into a [16][C] scratch (rows >= T zero),
// then a skinny tcgen05 GEMM with the weights as the M operand (128 x 16
// tiles), output transposed to [T][18D].
struct AdalnArgs {
  int C;                  // cond width (multiple of 64, <= 2816)
  int T;                  // timestep rows (1..16)
  int NW;                 // 18*D output channels (multiple of 128)
  int D;                  // residual width
  int chunk_lo, chunk_hi; // compute the table chunks [chunk_lo, chunk_hi) of every modality
  int max_ctas;           // 0: one CTA per SM; otherwise at most this many
  int l2_pf;              // stages of weight L2 prefetch ahead of the loads (0: none); set by the launcher
  const float* t_cond;    // [T][C]
  const __nv_bfloat16* bias;  // [NW] nullable (one block)
  __nv_bfloat16* out;     // [T][NW] (block b of a batch at out + b * out_block_stride)
  int n_blocks;           // blocks of a batched launch (1 otherwise)
  size_t out_block_stride;  // elements between the tables of consecutive blocks
  uint32_t* err;
};
// Weight tensor maps and biases of the blocks of one batched AdaLN-table
// launch (a kernel parameter; 64 maps are 8 KB).
constexpr int kAdalnBatch = 64;
template <int NM>
struct AdalnMaps {
  CUtensorMap w[NM];
  const __nv_bfloat16* bias[NM];
};
using AdalnBatchMaps = AdalnMaps<kAdalnBatch>;
cudaError_t launch_silu_rows(const float* t_cond, int T, int C, __nv_bfloat16* u, uint32_t* zero_words,
                             int n_zero_words, cudaStream_t stream);
cudaError_t launch_adaln_table(const CUtensorMap& tmW, const CUtensorMap& tmU, const AdalnArgs& a,
                               cudaStream_t stream);
// All chunks of the tables of a.n_blocks (<= kAdalnBatch) blocks in one launch.
cudaError_t launch_adaln_tables_batched(const AdalnBatchMaps& maps, const CUtensorMap& tmU, const AdalnArgs& a,
                                        cudaStream_t stream);
constexpr int kAdalnRows = 16;   // rows of the u scratch (T <= 16, zero padded)
// Widest AdaLN conditioning the library takes (the AdaLN-table kernel keeps
// all of u in shared memory; the configuration check, that kernel's shared
// memory plan and the no-allocation entry point's static scratch all derive
// from this one value).
constexpr int kMaxCondDim = 2816;

// ---------------------------------------------------------------------------
// attention (tcgen05 flash attention, one 128-row query tile per CTA)
// ---------------------------------------------------------------------------
struct AttnArgs {
  int S, H;
  __nv_bfloat16* o;       // [S][H*128]
  float* lse;             // [H][S] or null
  float scale_log2;       // log2(e) / sqrt(128)
  size_t o_elems, lse_elems;   // extents for the bounds-checked build
  uint32_t* err;
};
cudaError_t launch_attention(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                             const AttnArgs& a, cudaStream_t stream);

// ---------------------------------------------------------------------------
// row-wise kernels
// ---------------------------------------------------------------------------
struct ModulateArgs {
  int S, D, T;
  const __nv_bfloat16* x;
  const __nv_bfloat16* gain;
  const __nv_bfloat16* table;  // [3T][6][D]
  int chunk_shift, chunk_scale;
  const int32_t* tag;
  const int32_t* tidx;
  float eps;
  __nv_bfloat16* h;
  size_t x_elems, table_elems, h_elems;   // extents for the bounds-checked build
  uint32_t* err;
};
cudaError_t launch_modulate(const ModulateArgs& a, cudaStream_t stream);

struct RopeArgs {
  int S, H;
  __nv_bfloat16* q;
  __nv_bfloat16* k;
  int64_t row_stride, head_stride;
  const __nv_bfloat16* q_gain;
  const __nv_bfloat16* k_gain;
  const int32_t* pos;
  float eps;
  float omega[16];
  size_t qk_elems;        // elements from q (or k) to the end of its last row, for the bounds-checked build
  uint32_t* err;
};
// q and k maps: 3-D [S][H][128] views with the caller's strides, box {128, heads per unit, 1}
int rope_qknorm_heads_per_unit(int H);
int rope_qknorm_smem_bytes(int H);
cudaError_t launch_rope_qknorm(const CUtensorMap& tmq, const CUtensorMap& tmk, const RopeArgs& a, int num_sms,
                               cudaStream_t stream);

// token refiner: identity AdaLN table [3][6][D] and text / timestep-0 / zero-position metadata
cudaError_t launch_refiner_setup(int S, int D, __nv_bfloat16* table, int32_t* tag, int32_t* tidx, int32_t* pos,
                                 uint32_t* zero_words, int n_zero_words,
                                 cudaStream_t st);

// ---------------------------------------------------------------------------
// input side (k_input.cu)
// ---------------------------------------------------------------------------
struct InputProjArgs {
  int n, K, D, n_dst;
  const float* src;        // [n][K]
  const float* w;          // [D][K]
  const float* b;          // [D] or null
  const int32_t* dst;      // [n] destination rows
  __nv_bfloat16* out;      // [n_dst][D]
  uint32_t* err;
};
constexpr int kInputProjMaxK = 128;
cudaError_t launch_patch_pack(int C, int T, int H, int W, const float* src, float* dst, bool unpack,
                              cudaStream_t st);
cudaError_t launch_input_proj(const InputProjArgs& a, cudaStream_t st);
cudaError_t launch_index_copy(int n, int D, const __nv_bfloat16* src, const int32_t* dst, int n_dst,
                              __nv_bfloat16* out, uint32_t* err, cudaStream_t st);
cudaError_t launch_sinusoid(int T, const float* t, float* e_out, cudaStream_t st);
cudaError_t launch_rows_linear(int T, int K, int N, const float* in, const float* w, const float* b, int act,
                               float* out, cudaStream_t st);

// ---------------------------------------------------------------------------
// output side and sampler (k_output.cu)
// ---------------------------------------------------------------------------
struct OutputHeadArgs {
  int n_sel, S, T, D, P;
  const int32_t* rows;
  const int32_t* tidx;
  const __nv_bfloat16* x;   // [S][D]
  const float* table;       // [T][2][D]: shift, scale
  const float* w;           // [P][D]
  const float* b;           // [P] or null
  float* out;               // [n_sel][P]
  float eps;
  uint32_t* err;
};
constexpr int kOutputHeadMaxP = 128;
cudaError_t launch_sigma_grid(int n, float s, float* sigmas, int32_t* count, cudaStream_t st);
cudaError_t launch_ode_step(long long n, const float* xt, const float* v, float sigma, float sigma_next, float* out,
                            cudaStream_t st);
cudaError_t launch_noise_mix(long long n, const float* x0, const float* noise, float t, float* out, cudaStream_t st);
cudaError_t launch_select_rows(int n, const int32_t* tags, int tag, int32_t* rows, int32_t* count, cudaStream_t st);
constexpr int kFinalAdalnMaxTables = 4;
struct FinalAdalnArgs {
  int n_tables;                               // 1 .. kFinalAdalnMaxTables
  const float* w[kFinalAdalnMaxTables];       // [rows][C] each
  const float* b[kFinalAdalnMaxTables];       // [rows] or null
  float* out[kFinalAdalnMaxTables];           // [T][rows]
  const float* t_cond;                        // [T][C]
  int T, C, rows;                             // rows = 2D
};
cudaError_t launch_final_adaln(const FinalAdalnArgs& a, cudaStream_t st);
cudaError_t launch_output_head(const OutputHeadArgs& a, cudaStream_t st);

}  // namespace h3
