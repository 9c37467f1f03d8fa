// C ABI of libh3: argument validation (fail closed, before any launch), TMA
// tensor maps, the block's workspace plan and the stage composition.
#include "h3.h"
#include "h3_device.cuh"
#include "h3_internal.h"

#include <chrono>
#include <cmath>
#include <new>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <cstdlib>
#include <mutex>
#include <thread>

#include <cudaTypedefs.h>

namespace h3 {

// Device error words: [0] bits set by kernels on bad metadata or a wait that
// ran out, [1] the site of the first wait that ran out; read and cleared by
// h3_sync_check.
__device__ uint32_t g_error_word[2] = {0u, 0u};

namespace {
thread_local char g_info[512] = "";
constexpr int kMaxDevices = 64;
int g_sms[kMaxDevices] = {0};
uint32_t* g_err_ptr[kMaxDevices] = {nullptr};
std::mutex g_mu;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

int current_device() {
  int d = 0;
  cudaGetDevice(&d);
  return d < 0 || d >= kMaxDevices ? 0 : d;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  return g_encode;
}
}  // namespace

namespace {
char g_site[128] = "none";
std::mutex g_site_mu;

// Text of a site word (kernel id in the top byte; the low 24 bits are the
// barrier's shared-memory byte offset / 8, or kSiteStreamKFlag).
void note_error_site(uint32_t site) {
  static const char* const names[] = {"unknown", "gemm", "attention-1q", "attention-2q", "adaln-table",
                                      "rope-qknorm"};
  const uint32_t k = site >> 24, lo = site & 0xFFFFFFu;
  const char* kn = k < sizeof(names) / sizeof(names[0]) ? names[k] : "unknown";
  std::lock_guard<std::mutex> lk(g_site_mu);
  if (k & 0x80u)
    snprintf(g_site, sizeof(g_site), "bounds: access site %u, element offset %u from the buffer", k & 0x7Fu, lo);
  else if (site == 0)
    snprintf(g_site, sizeof(g_site), "timeout without a recorded site");
  else if (lo == kSiteStreamKFlag)
    snprintf(g_site, sizeof(g_site), "%s: stream-K partial-sum flag", kn);
  else
    snprintf(g_site, sizeof(g_site), "%s: mbarrier at shared offset %u", kn, lo * 8u);
}
}  // namespace

void set_kernel_info(const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_info, sizeof(g_info), fmt, ap);
  va_end(ap);
}

bool pdl_enabled() {
  static const bool on = [] {
    const char* e = getenv("H3_NO_PDL");
    return !(e && e[0] == '1');
  }();
  return on;
}

int num_sms() {
  const int d = current_device();
  if (!g_sms[d]) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, d);
    g_sms[d] = n > 0 ? n : 1;
  }
  return g_sms[d];
}

// If every TMEM kernel takes more than half of an SM's shared memory, no two
// of them (the same kernel or two different ones) fit on one SM together.
bool tmem_exclusive(int dyn_smem) {
  static int per_sm[kMaxDevices] = {0}, reserved[kMaxDevices] = {0};
  const int d = current_device();
  if (!per_sm[d]) {
    int p = 0, r = 0;
    if (cudaDeviceGetAttribute(&p, cudaDevAttrMaxSharedMemoryPerMultiprocessor, d) != cudaSuccess ||
        cudaDeviceGetAttribute(&r, cudaDevAttrReservedSharedMemoryPerBlock, d) != cudaSuccess || p <= 0) {
      cudaGetLastError();
      return false;
    }
    reserved[d] = r;
    per_sm[d] = p;
  }
  return 2 * (dyn_smem + reserved[d]) > per_sm[d];
}

uint32_t* device_error_word() {
  const int d = current_device();
  if (!g_err_ptr[d]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_error_word) == cudaSuccess) g_err_ptr[d] = static_cast<uint32_t*>(p);
  }
  return g_err_ptr[d];
}

bool make_tmap_2d(CUtensorMap* tm, const void* base, uint64_t rows, uint64_t cols, uint64_t ld,
                  uint32_t box_rows) {
  auto enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {ld * 2};
  const cuuint32_t box[2] = {64, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return enc(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_tmap_qkv(CUtensorMap* tm, const void* base, uint64_t n_rows, uint64_t n_heads, uint64_t row_stride,
                   uint64_t head_stride, uint32_t box_rows) {
  auto enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[3] = {128, n_heads, n_rows};
  const cuuint64_t strides[2] = {head_stride * 2, row_stride * 2};
  const cuuint32_t box[3] = {64, 1, box_rows};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// [S][H][128] bf16 view with the caller's row and head strides, unswizzled
// boxes of {128 channels, box_heads heads, 1 row}.
bool make_tmap_rope(CUtensorMap* tm, const void* base, uint64_t n_rows, uint64_t n_heads, uint64_t row_stride,
                    uint64_t head_stride, uint32_t box_heads) {
  auto enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[3] = {128, n_heads, n_rows};
  const cuuint64_t strides[2] = {head_stride * 2, row_stride * 2};
  const cuuint32_t box[3] = {128, box_heads, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace h3

using namespace h3;

// ===========================================================================
// validation helpers
// ===========================================================================
namespace {

inline bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool al16n(const void* p) { return p == nullptr || al16(p); }
inline size_t al256(size_t x) { return (x + 255) & ~size_t(255); }
constexpr int kMaxDevicesApi = 64;

h3_status check_cfg(const h3_block_config* c) {
  if (!c) return H3_ERR_NULL;
  if (c->head_dim != 128 || c->rope_freqs_per_axis != 16 || c->rope_channels != 96) return H3_ERR_UNSUPPORTED;
  if (c->dim < 64 || c->dim % 64 || c->dim > 8192) return H3_ERR_UNSUPPORTED;
  if (c->cond_dim < 64 || c->cond_dim % 64 || c->cond_dim > kMaxCondDim) return H3_ERR_UNSUPPORTED;
  if (c->ffn_dim < 128 || c->ffn_dim % 128) return H3_ERR_UNSUPPORTED;
  if (c->n_heads < 1 || c->n_heads > 1024) return H3_ERR_UNSUPPORTED;
  if (!(c->eps > 0.0f) || !std::isfinite(c->eps)) return H3_ERR_SHAPE;
  if (!(c->rope_theta > 1.0f) || !std::isfinite(c->rope_theta)) return H3_ERR_SHAPE;
  return H3_OK;
}

h3_status check_meta(const h3_packed_meta* m, bool need_tables) {
  if (!m) return H3_ERR_NULL;
  if (m->n_rows < 1) return H3_ERR_SHAPE;
  if (!m->token_tag || !m->timestep_index || !m->pos_thw) return H3_ERR_NULL;
  if (need_tables) {
    if (m->n_timesteps < 1 || m->n_timesteps > 16) return H3_ERR_UNSUPPORTED;
    if (!m->t_cond) return H3_ERR_NULL;
  }
  return H3_OK;
}

h3_status cuda_st(cudaError_t e) { return e == cudaSuccess ? H3_OK : H3_ERR_CUDA; }

void fill_omega(float* omega, float theta) {
  for (int i = 0; i < 16; ++i) omega[i] = (float)std::pow((double)theta, -(double)i / 16.0);
}

size_t adaln_scratch_bytes(const h3_block_config& c) { return al256((size_t)kAdalnRows * c.cond_dim * 2); }

struct WsLayout {
  size_t u, table, h, qkv, o, x1, sk_part, sk_flags, nrm_cnt, nrm_part, total;
  size_t zero_words;   // 32-bit words from sk_flags zeroed at the start of a block call
};
WsLayout ws_layout(const h3_block_config& c, int64_t S, int64_t T) {
  const size_t D = (size_t)c.dim, I = (size_t)c.n_heads * 128, F = (size_t)c.ffn_dim;
  WsLayout L{};
  size_t off = 0;
  L.u = off;     // bf16(SiLU(t_cond)), [16][C]
  off = al256(off + adaln_scratch_bytes(c));
  L.table = off;
  off = al256(off + (size_t)T * 18 * D * 2);
  L.h = off;
  off = al256(off + (size_t)S * D * 2);
  L.qkv = off;   // qkv [S][3I], later the SwiGLU activations [S][F]
  off = al256(off + (size_t)S * (3 * I > F ? 3 * I : F) * 2);
  L.o = off;
  off = al256(off + (size_t)S * I * 2);
  L.x1 = off;
  off = al256(off + (size_t)S * D * 2);
  L.sk_part = off;   // stream-K partial accumulators and flags of the residual GEMMs
  off = al256(off + gemm_sk_part_bytes());
  L.sk_flags = off;
  off = al256(off + gemm_sk_flag_words() * 4);
  // fused-norm counters (one per 256-row tile, zeroed with the flags) and
  // partial sums of squares (per row, two per 256-column tile)
  const size_t m_tiles = (size_t)((S + 255) / 256), n_tiles = (D + 255) / 256;
  L.nrm_cnt = off;
  off = al256(off + m_tiles * 4);
  L.zero_words = (L.nrm_cnt - L.sk_flags) / 4 + m_tiles;
  L.nrm_part = off;
  off = al256(off + m_tiles * 256 * 2 * n_tiles * 4);
  L.total = off;
  return L;
}

// ---------------------------------------------------------------------------
// stage launchers (arguments already validated)
// ---------------------------------------------------------------------------
// Table chunks [chunk_lo, chunk_hi) of every modality, from the SiLU rows u.
h3_status run_adaln_chunks(const h3_block_config& c, const void* w_ada, const void* b_ada, int T, void* out,
                           const void* u_scratch, int chunk_lo, int chunk_hi, int max_ctas, cudaStream_t st) {
  CUtensorMap tm, tu;
  if (!make_tmap_2d(&tm, w_ada, (uint64_t)18 * c.dim, (uint64_t)c.cond_dim, (uint64_t)c.cond_dim, 128) ||
      !make_tmap_2d(&tu, u_scratch, kAdalnRows, (uint64_t)c.cond_dim, (uint64_t)c.cond_dim, kAdalnRows))
    return H3_ERR_CUDA;
  AdalnArgs a{};
  a.C = c.cond_dim;
  a.T = T;
  a.NW = 18 * c.dim;
  a.D = c.dim;
  a.chunk_lo = chunk_lo;
  a.chunk_hi = chunk_hi;
  a.max_ctas = max_ctas;
  a.bias = static_cast<const __nv_bfloat16*>(b_ada);
  a.out = static_cast<__nv_bfloat16*>(out);
  a.err = device_error_word();
  return cuda_st(launch_adaln_table(tm, tu, a, st));
}

h3_status run_silu(const h3_block_config& c, const float* t_cond, int T, void* u_scratch, cudaStream_t st,
                   uint32_t* zero_words = nullptr, int n_zero_words = 0) {
  return cuda_st(launch_silu_rows(t_cond, T, c.cond_dim, static_cast<__nv_bfloat16*>(u_scratch), zero_words,
                                  n_zero_words, st));
}

h3_status run_adaln_table(const h3_block_config& c, const void* w_ada, const void* b_ada, const float* t_cond,
                          int T, void* out, void* u_scratch, cudaStream_t st) {
  h3_status s0 = run_silu(c, t_cond, T, u_scratch, st);
  if (s0 != H3_OK) return s0;
  // one launch over all six chunks (exact for every D, including D not a
  // multiple of 128 where a weight tile straddles two chunks)
  return run_adaln_chunks(c, w_ada, b_ada, T, out, u_scratch, 0, 6, 0, st);
}

h3_status run_modulate(const h3_block_config& c, const h3_packed_meta& m, const void* table, int branch,
                       const void* x, const void* g, void* h, cudaStream_t st) {
  ModulateArgs a{};
  a.S = m.n_rows;
  a.D = c.dim;
  a.T = m.n_timesteps;
  a.x = static_cast<const __nv_bfloat16*>(x);
  a.gain = static_cast<const __nv_bfloat16*>(g);
  a.table = static_cast<const __nv_bfloat16*>(table);
  a.chunk_shift = branch == 0 ? 0 : 3;
  a.chunk_scale = branch == 0 ? 1 : 4;
  a.tag = m.token_tag;
  a.tidx = m.timestep_index;
  a.x_elems = a.h_elems = (size_t)m.n_rows * c.dim;
  a.table_elems = (size_t)3 * m.n_timesteps * 6 * c.dim;
  a.eps = c.eps;
  a.h = static_cast<__nv_bfloat16*>(h);
  a.err = device_error_word();
  return cuda_st(launch_modulate(a, st));
}

void gemm_set_plan(GemmArgs& a, const GemmPlan& p) {
  a.b_rows = p.b_rows;
  a.nw1 = p.nw1;
  a.ncnt1 = p.ncnt1;
  a.nw2 = p.nw2;
}

// Stream-K fields of a launch with sk_lane pairs per row tile (see GemmArgs),
// or, with tail_units > 0, of a launch whose first dp tiles run whole and
// whose remaining tiles form one lane of tail_units pairs.
void gemm_set_sk(GemmArgs& a, int sk_lane, SkScratch* sk, int tail_units = 0, int dp = 0) {
  if (tail_units > 0) {
    a.sk_tail = 1;
    a.sk_dp = dp;
    a.sk_lane = tail_units;
    a.sk_units = tail_units;
    a.sk_iters = ((long long)a.num_m * a.num_n - dp) * a.num_k;
  } else {
    a.sk_lane = sk_lane;
    a.sk_units = a.num_m * sk_lane;
    a.sk_iters = (long long)a.num_n * a.num_k;
  }
  a.sk_part = sk->part;
  a.sk_flags = sk->flags;
  a.sk_epoch = ++sk->epoch;
  // H3_GEMM_L2HINT=0 turns the L2 eviction hints of stream-K launches off.
  // They serve the lanes of short documents (every row tile's lane streams
  // the same weight k-blocks while its pairs reread the activations); a tail
  // launch walks whole tiles first, as a plain launch does, and loads plainly.
  const char* h = getenv("H3_GEMM_L2HINT");
  a.l2_hint = (tail_units > 0 || (h && h[0] == '0')) ? 0 : 1;
  // H3_SK_FLAG_TEST=1 (tests of the failure path only): owners wait for a
  // flag value that no partial writer sets, so every owner's bounded wait
  // runs out and the launch reports H3_ERR_TIMEOUT through h3_sync_check
  // instead of producing its output; nothing traps or hangs.
  const char* t = getenv("H3_SK_FLAG_TEST");
  a.sk_wait = (t && t[0] == '1') ? (a.sk_epoch | 0x80000000u) : a.sk_epoch;
}

// The plan of a stream-K launch: whole-width 256-column tiles.
GemmPlan sk_plan(int epi, int N, int H, int F) {
  GemmPlan p{};
  p.bn = 256;
  p.num_n = gemm_num_n(epi, 256, N, H, F);
  p.b_rows = gemm_b_box_rows(epi, 256);
  return p;
}

void gemm_common(GemmArgs& a, int M, int K, int num_n) {
  a.M = M;
  a.K = K;
  a.num_m = gemm_m_tiles(M);
  a.num_n = num_n;
  a.num_k = K / 64;
  a.err = device_error_word();
}

h3_status run_qkv(const h3_block_config& c, const h3_packed_meta& m, const void* h, const void* w_qkv,
                  const void* b_qkv, const void* qg, const void* kg, void* out, cudaStream_t st,
                  int max_ctas = 0) {
  const int S = m.n_rows, D = c.dim, H = c.n_heads;
  const GemmPlan pl = gemm_plan(EPI_QKV, S, 3 * H * 128, H, 0);
  CUtensorMap tA, tB;
  if (!make_tmap_2d(&tA, h, S, D, D, 128) ||
      !make_tmap_2d(&tB, w_qkv, (uint64_t)3 * H * 128, D, D, (uint32_t)pl.b_rows))
    return H3_ERR_CUDA;
  GemmArgs a{};
  gemm_common(a, S, D, pl.num_n);
  gemm_set_plan(a, pl);
  a.out = static_cast<__nv_bfloat16*>(out);
  a.ldo = 3 * H * 128;
  a.bias = static_cast<const __nv_bfloat16*>(b_qkv);
  a.H = H;
  a.q_gain = static_cast<const __nv_bfloat16*>(qg);
  a.k_gain = static_cast<const __nv_bfloat16*>(kg);
  a.pos = m.pos_thw;
  a.eps = c.eps;
  a.max_ctas = max_ctas;
  fill_omega(a.omega, c.rope_theta);
  return cuda_st(launch_gemm(EPI_QKV, pl.bn, tA, tB, a, st));
}

h3_status run_attention(int S, int H, const void* q, const void* k, const void* v, int64_t rs, int64_t hs,
                        void* o, float* lse, cudaStream_t st) {
  CUtensorMap tq, tk, tv;
  if (!make_tmap_qkv(&tq, q, S, H, rs, hs, 128) || !make_tmap_qkv(&tk, k, S, H, rs, hs, 128) ||
      !make_tmap_qkv(&tv, v, S, H, rs, hs, 128))
    return H3_ERR_CUDA;
  AttnArgs a{};
  a.S = S;
  a.H = H;
  a.o = static_cast<__nv_bfloat16*>(o);
  a.lse = lse;
  a.o_elems = (size_t)S * H * 128;
  a.lse_elems = lse ? (size_t)H * S : 0;
  a.scale_log2 = (float)(1.4426950408889634 / std::sqrt(128.0));
  a.err = device_error_word();
  return cuda_st(launch_attention(tq, tk, tv, a, st));
}

// sk: stream-K scratch of the calling block (flags zeroed by its first
// kernel); null for the stand-alone stage, which runs whole tiles only.
// (The QKV and FC1 GEMMs run whole tiles: at 256 rows, where their last
// wave is short, stream-K measured no faster over the refiner pass.)
// The norm + modulation a residual GEMM may emit as well (norm2 after the O
// projection): the output h, its gain and table chunks.
struct NormFuse {
  void* h;
  const void* gain;
  int shift, scale;
};

// Fuse the following norm into a stream-K residual GEMM: off by default,
// H3_NORM_FUSE=1 in the environment turns it on.  Measured on GB300 it loses:
// the O projection waits for the last owner of each row tile before any row
// can be normed, which costs more than the separate norm2 launch it saves
// (505 rows: O 60.7 -> 75.6 us against norm2 8.6 -> 0; block 0.386 -> 0.398
// ms; 1824 rows: 1.081 -> 1.122 ms).
bool norm_fuse_enabled() {
  const char* e = getenv("H3_NORM_FUSE");
  return e && e[0] == '1';
}

// A stream-K residual GEMM with lanes of sk_lane pairs can carry the norm
// when each pair's run spans few enough tiles (every epilogue warp keeps
// the four tiles it may own).
bool norm_fuse_fits(int sk_lane, int num_n, int num_k) {
  return sk_lane > 0 && norm_fuse_enabled() && (long long)num_n * num_k / sk_lane / num_k + 2 <= 4;
}

// Whether the block's O projection carries norm2 at S rows on this device.
bool o_norm_fused(const h3_block_config& c, int S) {
  const int I = c.n_heads * 128;
  return norm_fuse_fits(gemm_sk_lane(S, c.dim, I, 256, 0), (c.dim + 255) / 256, I / 64);
}

h3_status run_resid_gemm(const h3_block_config& c, const h3_packed_meta& m, const void* table, int chunk,
                         const void* act, int K, const void* w, const void* b, const void* x, void* out,
                         cudaStream_t st, SkScratch* sk = nullptr, const NormFuse* nf = nullptr,
                         bool* fused = nullptr) {
  if (fused) *fused = false;
  const int S = m.n_rows, D = c.dim;
  GemmPlan pl = gemm_plan(EPI_RESID, S, D, 0, 0);
  // stream-K: lanes of pairs per row tile for short documents; for long ones
  // whole tiles with the last waves' k-blocks shared out over every pair
  // (H3_GEMM_SK_TAIL=n forces the second form with n pairs)
  int tail_units = 0, dp = -1;
  if (sk) dp = gemm_sk_tail(S, D, K, 256, &tail_units);
  const bool forced_tail = getenv("H3_GEMM_SK_TAIL") != nullptr;
  const int sk_lane = (sk && !(forced_tail && dp >= 0)) ? gemm_sk_lane(S, D, K, 256, 0) : 0;
  if (sk_lane > 0 || dp < 0) tail_units = 0;
  if (sk_lane > 0 || tail_units > 0) pl = sk_plan(EPI_RESID, D, 0, 0);   // whole-width tiles, k-blocks shared out
  CUtensorMap tA, tB;
  if (!make_tmap_2d(&tA, act, S, K, K, 128) || !make_tmap_2d(&tB, w, D, K, K, (uint32_t)pl.b_rows))
    return H3_ERR_CUDA;
  GemmArgs a{};
  gemm_common(a, S, K, pl.num_n);
  gemm_set_plan(a, pl);
  a.out = static_cast<__nv_bfloat16*>(out);
  a.ldo = D;
  a.bias = static_cast<const __nv_bfloat16*>(b);
  a.n_valid = D;
  a.resid = static_cast<const __nv_bfloat16*>(x);
  a.ldr = D;
  a.table = static_cast<const __nv_bfloat16*>(table);
  a.D = D;
  a.chunk = chunk;
  a.T = m.n_timesteps;
  a.tag = m.token_tag;
  a.tidx = m.timestep_index;
  if (sk_lane > 0) gemm_set_sk(a, sk_lane, sk);
  else if (tail_units > 0) gemm_set_sk(a, 0, sk, tail_units, dp);
  // the fused norm needs every pair resident (stream-K) and runs of at most
  // two whole tiles plus a partial piece (each warp keeps four owned tiles)
  if (nf && sk->nrm_cnt && norm_fuse_fits(sk_lane, a.num_n, a.num_k)) {
    a.nrm_h = static_cast<__nv_bfloat16*>(nf->h);
    a.nrm_gain = static_cast<const __nv_bfloat16*>(nf->gain);
    a.nrm_shift = nf->shift;
    a.nrm_scale = nf->scale;
    a.nrm_part = sk->nrm_part;
    a.nrm_cnt = sk->nrm_cnt;
    a.nrm_target = (++sk->nrm_launches) * 16u * (uint32_t)a.num_n;
    if (fused) *fused = true;
  }
  return cuda_st(launch_gemm(EPI_RESID, pl.bn, tA, tB, a, st));
}

h3_status run_ffn_up(const h3_block_config& c, int S, const void* h, const void* w1, const void* b1, void* out,
                     cudaStream_t st) {
  const int D = c.dim, F = c.ffn_dim;
  const GemmPlan pl = gemm_plan(EPI_SWIGLU, S, 2 * F, 0, F);
  CUtensorMap tA, tB;
  if (!make_tmap_2d(&tA, h, S, D, D, 128) || !make_tmap_2d(&tB, w1, (uint64_t)2 * F, D, D, (uint32_t)pl.b_rows))
    return H3_ERR_CUDA;
  GemmArgs a{};
  gemm_common(a, S, D, pl.num_n);
  gemm_set_plan(a, pl);
  a.out = static_cast<__nv_bfloat16*>(out);
  a.ldo = F;
  a.bias = static_cast<const __nv_bfloat16*>(b1);
  a.F = F;
  return cuda_st(launch_gemm(EPI_SWIGLU, pl.bn, tA, tB, a, st));
}

h3_status check_block_weights(const h3_block_weights* w) {
  if (!w) return H3_ERR_NULL;
  if (!w->w_ada || !w->norm1_g || !w->norm2_g || !w->w_qkv || !w->q_norm_g || !w->k_norm_g || !w->w_o ||
      !w->w_fc1 || !w->w_fc2)
    return H3_ERR_NULL;
  const void* req[] = {w->w_ada, w->norm1_g, w->norm2_g, w->w_qkv, w->q_norm_g, w->k_norm_g,
                       w->w_o, w->w_fc1, w->w_fc2};
  for (const void* p : req)
    if (!al16(p)) return H3_ERR_ALIGN;
  const void* opt[] = {w->b_ada, w->b_qkv, w->b_o, w->b_fc1, w->b_fc2};
  for (const void* p : opt)
    if (!al16n(p)) return H3_ERR_ALIGN;
  return H3_OK;
}

// Table chunks of one block computed on the caller's stream when the rest
// goes to the side stream: shift, scale and gate of the attention half.
constexpr int kMainChunks = 3;

// SMs for the AdaLN chunks 3-5 on the side stream, 0 when the table is not
// split: the split needs D a multiple of 128 (whole chunks per weight tile)
// and pays only when the QKV GEMM leaves at least 8 SMs free at its wave
// count (short documents); otherwise every SM already has GEMM work.
int adaln_side_ctas(const h3_block_config& c, int S) {
  if (c.dim % 128) return 0;
  const int sms = num_sms(), H = c.n_heads, I = H * 128;
  const GemmPlan pl = gemm_plan(EPI_QKV, S, 3 * I, H, 0);
  const int slots = gemm_pair_slots();
  if (slots < 1 || sms < 8) return 0;
  const long long tiles = (long long)gemm_m_tiles(S) * pl.num_n;
  const long long waves = (tiles + slots - 1) / slots;
  const int need = 2 * (int)((tiles + waves - 1) / waves);   // fewest CTAs (pairs x 2) with the same wave count
  return sms - need >= 8 ? sms - need : 0;
}

// A library-owned stream per device for work that overlaps the caller's
// stream inside one call (joined back by events before the call returns).
cudaStream_t side_stream() {
  static cudaStream_t streams[kMaxDevicesApi] = {nullptr};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevicesApi) return nullptr;
  std::lock_guard<std::mutex> lk(mu);
  if (!streams[dev] && cudaStreamCreateWithFlags(&streams[dev], cudaStreamNonBlocking) != cudaSuccess)
    streams[dev] = nullptr;
  return streams[dev];
}

// x_ready: when not null, an event the caller's stream waits for before the
// first kernel that reads x_in (norm1); the AdaLN table does not read it.
// A library-owned stream per device for the host-to-device copy of a block
// input that overlaps the AdaLN table (joined by an event before norm1).
cudaStream_t copy_stream() {
  static cudaStream_t streams[kMaxDevicesApi] = {nullptr};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevicesApi) return nullptr;
  std::lock_guard<std::mutex> lk(mu);
  if (!streams[dev] && cudaStreamCreateWithFlags(&streams[dev], cudaStreamNonBlocking) != cudaSuccess)
    streams[dev] = nullptr;
  return streams[dev];
}

// table_pre: the block's AdaLN table computed beforehand (a chain's batched
// tables); the block then starts at norm1.  sk_chain: stream-K scratch whose
// flags the chain zeroed once and whose epoch runs on across its blocks.
h3_status block_impl(const h3_block_config* cfg, const h3_block_weights* w, const h3_packed_meta* meta,
                     const void* x_in, void* x_out, void* ws, size_t ws_bytes, cudaStream_t st,
                     void* const* events, int n_events, cudaEvent_t x_ready = nullptr,
                     const void* table_pre = nullptr, SkScratch* sk_chain = nullptr) {
  const int S = meta->n_rows, T = meta->n_timesteps;
  const WsLayout L = ws_layout(*cfg, S, T);
  uint8_t* base = static_cast<uint8_t*>(ws);
  void* u = base + L.u;
  void* table = table_pre ? const_cast<void*>(table_pre) : base + L.table;
  void* h = base + L.h;
  void* qkv = base + L.qkv;
  void* o = base + L.o;
  void* x1 = base + L.x1;
  SkScratch sk_own{reinterpret_cast<float*>(base + L.sk_part), reinterpret_cast<uint32_t*>(base + L.sk_flags), 0,
                   reinterpret_cast<float*>(base + L.nrm_part), reinterpret_cast<uint32_t*>(base + L.nrm_cnt), 0};
  SkScratch& sk = sk_chain ? *sk_chain : sk_own;
  const int I = cfg->n_heads * 128;
  int stage = 0;
  auto mark = [&]() -> h3_status {
    if (events && stage < n_events && events[stage]) {
      if (cudaEventRecord(static_cast<cudaEvent_t>(events[stage]), st) != cudaSuccess) return H3_ERR_CUDA;
    }
    ++stage;
    return H3_OK;
  };
  h3_status s;
#define H3_TRY(expr)            \
  if ((s = (expr)) != H3_OK) return s; \
  if ((s = mark()) != H3_OK) return s;
  // Stage 0, the AdaLN table.  norm1 reads chunks 0-1 (shift_msa,
  // scale_msa) and the O projection chunk 2 (gate_msa); chunks 3-5 are first
  // read by norm2.  Chunks 0-2 run on the caller's stream; chunks 3-5 (half
  // of the weight stream) run on the side stream on the SMs that the QKV
  // GEMM's wave count leaves free, and the caller's stream waits for them
  // before norm2.
  if (!table_pre) {
    s = run_silu(*cfg, meta->t_cond, T, u, st, sk.flags, (int)L.zero_words);
    if (s != H3_OK) return s;
  }
  const int side_ctas = table_pre ? 0 : adaln_side_ctas(*cfg, S);
  cudaStream_t side = side_ctas > 0 ? side_stream() : nullptr;
  cudaEvent_t ev_a = nullptr, ev_b = nullptr;
  struct EventGuard {
    cudaEvent_t* e[2];
    ~EventGuard() {
      for (cudaEvent_t* p : e)
        if (*p) cudaEventDestroy(*p);
    }
  } guard{{&ev_a, &ev_b}};
  if (side) {
    if (cudaEventCreateWithFlags(&ev_a, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&ev_b, cudaEventDisableTiming) != cudaSuccess)
      return H3_ERR_CUDA;
  }
  int qkv_ctas = 0;
  if (side) {
    qkv_ctas = num_sms() - side_ctas;
    if ((s = run_adaln_chunks(*cfg, w->w_ada, w->b_ada, T, table, u, 0, kMainChunks, 0, st)) != H3_OK) return s;
    if (cudaEventRecord(ev_a, st) != cudaSuccess || cudaStreamWaitEvent(side, ev_a, 0) != cudaSuccess)
      return H3_ERR_CUDA;
    if (events && n_events > 8 && events[8] &&
        cudaEventRecord(static_cast<cudaEvent_t>(events[8]), side) != cudaSuccess)
      return H3_ERR_CUDA;
    // (Two side launches, the gate chunk first so that the O projection
    // would wait for it alone, measured slower at 505 rows: the QKV GEMM
    // beside them took 133 instead of 102 us.  With the second launched
    // after the QKV GEMM and without programmatic early start, the GEMM
    // kept its 102 us, but the plain block took 0.408 instead of 0.387 ms:
    // each cross-stream wait ends the programmatic overlap of the kernel
    // after it.  Hence one side launch, and the gate on this stream.)
    if ((s = run_adaln_chunks(*cfg, w->w_ada, w->b_ada, T, table, u, kMainChunks, 6, side_ctas, side)) != H3_OK)
      return s;
    if (events && n_events > 9 && events[9] &&
        cudaEventRecord(static_cast<cudaEvent_t>(events[9]), side) != cudaSuccess)
      return H3_ERR_CUDA;
    if (cudaEventRecord(ev_b, side) != cudaSuccess) return H3_ERR_CUDA;
  } else if (!table_pre) {
    if ((s = run_adaln_chunks(*cfg, w->w_ada, w->b_ada, T, table, u, 0, 6, 0, st)) != H3_OK) return s;
  }
  if ((s = mark()) != H3_OK) return s;
  if (x_ready && cudaStreamWaitEvent(st, x_ready, 0) != cudaSuccess) return H3_ERR_CUDA;
  H3_TRY(run_modulate(*cfg, *meta, table, 0, x_in, w->norm1_g, h, st));
  H3_TRY(run_qkv(*cfg, *meta, h, w->w_qkv, w->b_qkv, w->q_norm_g, w->k_norm_g, qkv, st, qkv_ctas));
  {
    const __nv_bfloat16* q = static_cast<const __nv_bfloat16*>(qkv);
    H3_TRY(run_attention(S, cfg->n_heads, q, q + 128, q + 256, 3 * I, 384, o, nullptr, st));
  }
  // norm2 + modulation rides in the O projection's epilogue when that GEMM
  // runs stream-K and H3_NORM_FUSE is set (it then needs chunks 3-4 before
  // the O projection); otherwise it is its own kernel
  const bool may_fuse = norm_fuse_enabled();
  if (side && may_fuse && cudaStreamWaitEvent(st, ev_b, 0) != cudaSuccess) return H3_ERR_CUDA;
  bool fused = false;
  const NormFuse nf{h, w->norm2_g, 3, 4};
  H3_TRY(run_resid_gemm(*cfg, *meta, table, 2, o, I, w->w_o, w->b_o, x_in, x1, st, &sk, &nf, &fused));
  if (fused) {
    if ((s = mark()) != H3_OK) return s;
  } else {
    if (side && !may_fuse && cudaStreamWaitEvent(st, ev_b, 0) != cudaSuccess) return H3_ERR_CUDA;
    H3_TRY(run_modulate(*cfg, *meta, table, 1, x1, w->norm2_g, h, st));
  }
  H3_TRY(run_ffn_up(*cfg, S, h, w->w_fc1, w->b_fc1, qkv, st));
  H3_TRY(run_resid_gemm(*cfg, *meta, table, 5, qkv, cfg->ffn_dim, w->w_fc2, w->b_fc2, x1, x_out, st, &sk));
#undef H3_TRY
  return H3_OK;
}

// A chain computes the AdaLN tables of all its blocks up front, in one
// launch per kAdalnBatch blocks, where a block would get no overlap from the
// side stream (the QKV GEMM keeps every SM busy); the tables then follow the
// block workspace.  Otherwise each block computes its own table.
bool chain_batches_tables(const h3_block_config& c, int n_blocks, int S) {
  return n_blocks > 1 && adaln_side_ctas(c, S) == 0;
}
size_t chain_table_bytes(const h3_block_config& c, int64_t T) { return al256((size_t)T * 18 * c.dim * 2); }
size_t chain_ws_bytes(const h3_block_config& c, int n_blocks, int64_t S, int64_t T) {
  size_t n = ws_layout(c, S, T).total;
  if (chain_batches_tables(c, n_blocks, (int)S)) n += (size_t)n_blocks * chain_table_bytes(c, T);
  return n;
}

// The blocks w[0 .. n_blocks) in order: x_in -> x_out (block b > 0 reads
// x_out); x_ready as for block_impl (first block only).
h3_status chain_impl(const h3_block_config* cfg, int n_blocks, const h3_block_weights* w,
                     const h3_packed_meta* meta, const void* x_in, void* x_out, void* ws, size_t ws_bytes,
                     cudaStream_t st, cudaEvent_t x_ready = nullptr) {
  const int S = meta->n_rows, T = meta->n_timesteps;
  if (!chain_batches_tables(*cfg, n_blocks, S)) {
    for (int b = 0; b < n_blocks; ++b) {
      h3_status s = block_impl(cfg, &w[b], meta, b == 0 ? x_in : x_out, x_out, ws, ws_bytes, st, nullptr, 0,
                               b == 0 ? x_ready : nullptr);
      if (s != H3_OK) return s;
    }
    return H3_OK;
  }
  const WsLayout L = ws_layout(*cfg, S, T);
  uint8_t* base = static_cast<uint8_t*>(ws);
  uint8_t* tables = base + L.total;
  const size_t tb = chain_table_bytes(*cfg, T);
  SkScratch sk{reinterpret_cast<float*>(base + L.sk_part), reinterpret_cast<uint32_t*>(base + L.sk_flags), 0,
               reinterpret_cast<float*>(base + L.nrm_part), reinterpret_cast<uint32_t*>(base + L.nrm_cnt), 0};
  // u = bf16(SiLU(t_cond)) once (the blocks share t_cond); the same launch
  // zeroes the stream-K flags and fused-norm counters, whose epochs and
  // counts then run on across the chain
  h3_status s = run_silu(*cfg, meta->t_cond, T, base + L.u, st, sk.flags, (int)L.zero_words);
  if (s != H3_OK) return s;
  CUtensorMap tu;
  if (!make_tmap_2d(&tu, base + L.u, kAdalnRows, (uint64_t)cfg->cond_dim, (uint64_t)cfg->cond_dim, kAdalnRows))
    return H3_ERR_CUDA;
  static thread_local AdalnBatchMaps maps;   // 8 KB: kept off the stack
  for (int b0 = 0; b0 < n_blocks; b0 += kAdalnBatch) {
    const int nb = n_blocks - b0 < kAdalnBatch ? n_blocks - b0 : kAdalnBatch;
    for (int i = 0; i < nb; ++i) {
      if (!make_tmap_2d(&maps.w[i], w[b0 + i].w_ada, (uint64_t)18 * cfg->dim, (uint64_t)cfg->cond_dim,
                        (uint64_t)cfg->cond_dim, 128))
        return H3_ERR_CUDA;
      maps.bias[i] = static_cast<const __nv_bfloat16*>(w[b0 + i].b_ada);
    }
    AdalnArgs a{};
    a.C = cfg->cond_dim;
    a.T = T;
    a.NW = 18 * cfg->dim;
    a.D = cfg->dim;
    a.chunk_lo = 0;
    a.chunk_hi = 6;
    a.out = reinterpret_cast<__nv_bfloat16*>(tables + (size_t)b0 * tb);
    a.n_blocks = nb;
    a.out_block_stride = tb / 2;
    a.err = device_error_word();
    if ((s = cuda_st(launch_adaln_tables_batched(maps, tu, a, st))) != H3_OK) return s;
  }
  for (int b = 0; b < n_blocks; ++b) {
    s = block_impl(cfg, &w[b], meta, b == 0 ? x_in : x_out, x_out, ws, ws_bytes, st, nullptr, 0,
                   b == 0 ? x_ready : nullptr, tables + (size_t)b * tb, &sk);
    if (s != H3_OK) return s;
  }
  return H3_OK;
}

h3_status check_block_args(const h3_block_config* cfg, const h3_block_weights* w, const h3_packed_meta* meta,
                           const void* x_in, void* x_out, void* ws, size_t ws_bytes) {
  h3_status s;
  if ((s = check_cfg(cfg)) != H3_OK) return s;
  if ((s = check_meta(meta, true)) != H3_OK) return s;
  if ((s = check_block_weights(w)) != H3_OK) return s;
  if (!x_in || !x_out || !ws) return H3_ERR_NULL;
  if (!al16(x_in) || !al16(x_out) || (reinterpret_cast<uintptr_t>(ws) & 255u)) return H3_ERR_ALIGN;
  if (ws_bytes < ws_layout(*cfg, meta->n_rows, meta->n_timesteps).total) return H3_ERR_WORKSPACE;
  return H3_OK;
}

// ---------------------------------------------------------------------------
// Scratch of h3_adaln_table_noalloc: the bf16 SiLU rows [16][cond_dim] live in
// a file-scope device array instead of caller memory.  Every GPU that loads
// the library holds it (16 x 2816 x 2 = 90,112 bytes) until the process exits.
// Host code may not pass the array's name to a kernel (on the host it is only
// a stand-in symbol): its device address is looked up once per device.
// ---------------------------------------------------------------------------
constexpr int kNoAllocMaxCond = kMaxCondDim;   // every width the configuration check accepts
void* g_noalloc_scratch[kMaxDevicesApi] = {nullptr};
std::mutex g_noalloc_mu;

}  // namespace

static __device__ __align__(256) __nv_bfloat16 h3_noalloc_silu_rows[kAdalnRows * kNoAllocMaxCond];

namespace {
// Device address of the array for the current device; the first call on a
// device (made with that device current) performs the lookup.
h3_status noalloc_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return H3_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevicesApi) return H3_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (!g_noalloc_scratch[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, h3_noalloc_silu_rows) != cudaSuccess || p == nullptr) return H3_ERR_CUDA;
    g_noalloc_scratch[dev] = p;
  }
  *out = g_noalloc_scratch[dev];
  return H3_OK;
}
}  // namespace

// ===========================================================================
// exported C ABI
// ===========================================================================
extern "C" {

size_t h3_block_workspace_bytes(const h3_block_config* cfg, int32_t n_rows, int32_t n_timesteps) {
  if (check_cfg(cfg) != H3_OK || n_rows < 1 || n_timesteps < 1 || n_timesteps > 16) return 0;
  return ws_layout(*cfg, n_rows, n_timesteps).total;
}

int32_t h3_blocks_kernel_count(const h3_block_config* cfg, int32_t n_blocks, int32_t n_rows) {
  if (check_cfg(cfg) != H3_OK || n_blocks < 1 || n_rows < 1) return 0;
  const bool side = adaln_side_ctas(*cfg, n_rows) > 0;
  const bool batched = chain_batches_tables(*cfg, n_blocks, n_rows);
  // norm1, QKV, attention, O, norm2 (unless fused), FC1, FC2
  const int stages = 7 - (o_norm_fused(*cfg, n_rows) ? 1 : 0);
  if (batched) return 1 + (n_blocks + kAdalnBatch - 1) / kAdalnBatch + n_blocks * stages;
  return n_blocks * (1 + (side ? 2 : 1) + stages);
}

int32_t h3_block_adaln_side_ctas(const h3_block_config* cfg, int32_t n_rows) {
  if (check_cfg(cfg) != H3_OK || n_rows < 1) return 0;
  return adaln_side_ctas(*cfg, n_rows);
}

h3_status h3_block_forward(const h3_block_config* cfg, const h3_block_weights* w, const h3_packed_meta* meta,
                           const void* x_in, void* x_out, void* workspace, size_t ws_bytes,
                           cudaStream_t stream) {
  h3_status s = check_block_args(cfg, w, meta, x_in, x_out, workspace, ws_bytes);
  if (s != H3_OK) return s;
  return block_impl(cfg, w, meta, x_in, x_out, workspace, ws_bytes, stream, nullptr, 0);
}

// Staging for h3_block_forward_host, after the block workspace: x, y, the
// three metadata arrays and t_cond.
struct HostStaging {
  size_t x, y, tag, tidx, pos, tcond, total;
};
HostStaging host_staging(const h3_block_config& c, int n_blocks, int64_t S, int64_t T) {
  HostStaging H{};
  size_t off = chain_ws_bytes(c, n_blocks, S, T);
  H.x = off;
  off = al256(off + (size_t)S * c.dim * 2);
  H.y = off;
  off = al256(off + (size_t)S * c.dim * 2);
  H.tag = off;
  off = al256(off + (size_t)S * 4);
  H.tidx = off;
  off = al256(off + (size_t)S * 4);
  H.pos = off;
  off = al256(off + (size_t)S * 12);
  H.tcond = off;
  off = al256(off + (size_t)T * c.cond_dim * 4);
  H.total = off;
  return H;
}

size_t h3_block_host_workspace_bytes(const h3_block_config* cfg, int32_t n_rows, int32_t n_timesteps) {
  if (check_cfg(cfg) != H3_OK || n_rows < 1 || n_timesteps < 1 || n_timesteps > 16) return 0;
  return host_staging(*cfg, 1, n_rows, n_timesteps).total;
}

size_t h3_blocks_host_workspace_bytes(const h3_block_config* cfg, int32_t n_blocks, int32_t n_rows,
                                      int32_t n_timesteps) {
  if (check_cfg(cfg) != H3_OK || n_blocks < 1 || n_rows < 1 || n_timesteps < 1 || n_timesteps > 16) return 0;
  return host_staging(*cfg, n_blocks, n_rows, n_timesteps).total;
}

size_t h3_blocks_workspace_bytes(const h3_block_config* cfg, int32_t n_blocks, int32_t n_rows, int32_t n_timesteps) {
  if (check_cfg(cfg) != H3_OK || n_blocks < 1 || n_rows < 1 || n_timesteps < 1 || n_timesteps > 16) return 0;
  return chain_ws_bytes(*cfg, n_blocks, n_rows, n_timesteps);
}

// The blocks w[0 .. n_blocks) from and to host memory through the staging.
static h3_status host_forward(const h3_block_config* cfg, int32_t n_blocks, const h3_block_weights* w,
                              const h3_packed_meta* meta_host, const void* x_host, void* y_host, void* workspace,
                              size_t ws_bytes, cudaStream_t stream) {
  h3_status s = check_cfg(cfg);
  if (s != H3_OK) return s;
  if (!w) return H3_ERR_NULL;
  if (n_blocks < 1) return H3_ERR_SHAPE;
  if ((s = check_meta(meta_host, true)) != H3_OK) return s;
  for (int b = 0; b < n_blocks; ++b)
    if ((s = check_block_weights(&w[b])) != H3_OK) return s;
  if (!x_host || !y_host || !workspace) return H3_ERR_NULL;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return H3_ERR_ALIGN;
  const int S = meta_host->n_rows, T = meta_host->n_timesteps;
  const HostStaging H = host_staging(*cfg, n_blocks, S, T);
  if (ws_bytes < H.total) return H3_ERR_WORKSPACE;
  uint8_t* base = static_cast<uint8_t*>(workspace);
  const size_t xb = (size_t)S * cfg->dim * 2;
  // One copy per host buffer.  The metadata go first on the caller's
  // stream; x goes on the library's copy stream, which starts after the
  // caller's earlier work (that may still use the staging) and which norm1
  // waits for, so that the copy overlaps the AdaLN table.
  const struct {
    size_t off;
    const void* src;
    size_t bytes;
  } in[4] = {{H.tag, meta_host->token_tag, (size_t)S * 4},
             {H.tidx, meta_host->timestep_index, (size_t)S * 4},
             {H.pos, meta_host->pos_thw, (size_t)S * 12},
             {H.tcond, meta_host->t_cond, (size_t)T * cfg->cond_dim * 4}};
  struct EventGuard {
    cudaEvent_t ev[2] = {nullptr, nullptr};
    ~EventGuard() {
      for (cudaEvent_t e : ev)
        if (e) cudaEventDestroy(e);
    }
  } guard;
  cudaStream_t cs = copy_stream();
  if (cs) {
    for (cudaEvent_t& e : guard.ev)
      if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) return H3_ERR_CUDA;
    if (cudaEventRecord(guard.ev[0], stream) != cudaSuccess || cudaStreamWaitEvent(cs, guard.ev[0], 0) != cudaSuccess ||
        cudaMemcpyAsync(base + H.x, x_host, xb, cudaMemcpyHostToDevice, cs) != cudaSuccess ||
        cudaEventRecord(guard.ev[1], cs) != cudaSuccess)
      return H3_ERR_CUDA;
  } else if (cudaMemcpyAsync(base + H.x, x_host, xb, cudaMemcpyHostToDevice, stream) != cudaSuccess) {
    return H3_ERR_CUDA;
  }
  for (const auto& c : in)
    if (cudaMemcpyAsync(base + c.off, c.src, c.bytes, cudaMemcpyHostToDevice, stream) != cudaSuccess)
      return H3_ERR_CUDA;
  const h3_packed_meta m{S, T, reinterpret_cast<const int32_t*>(base + H.tag),
                         reinterpret_cast<const int32_t*>(base + H.tidx), reinterpret_cast<const int32_t*>(base + H.pos),
                         reinterpret_cast<const float*>(base + H.tcond)};
  if ((s = chain_impl(cfg, n_blocks, w, &m, base + H.x, base + H.y, workspace, ws_bytes, stream, guard.ev[1])) !=
      H3_OK)
    return s;
  return cudaMemcpyAsync(y_host, base + H.y, xb, cudaMemcpyDeviceToHost, stream) == cudaSuccess ? H3_OK
                                                                                                : H3_ERR_CUDA;
}

h3_status h3_block_forward_host(const h3_block_config* cfg, const h3_block_weights* w,
                                const h3_packed_meta* meta_host, const void* x_host, void* y_host, void* workspace,
                                size_t ws_bytes, cudaStream_t stream) {
  return host_forward(cfg, 1, w, meta_host, x_host, y_host, workspace, ws_bytes, stream);
}

h3_status h3_blocks_forward_host(const h3_block_config* cfg, int32_t n_blocks, const h3_block_weights* w,
                                 const h3_packed_meta* meta_host, const void* x_host, void* y_host,
                                 void* workspace, size_t ws_bytes, cudaStream_t stream) {
  return host_forward(cfg, n_blocks, w, meta_host, x_host, y_host, workspace, ws_bytes, stream);
}

h3_status h3_block_forward_profiled(const h3_block_config* cfg, const h3_block_weights* w,
                                    const h3_packed_meta* meta, const void* x_in, void* x_out, void* workspace,
                                    size_t ws_bytes, cudaStream_t stream, void* const* events,
                                    int32_t n_events) {
  h3_status s = check_block_args(cfg, w, meta, x_in, x_out, workspace, ws_bytes);
  if (s != H3_OK) return s;
  if (n_events < 0) return H3_ERR_SHAPE;
  return block_impl(cfg, w, meta, x_in, x_out, workspace, ws_bytes, stream, events, n_events);
}

h3_status h3_blocks_forward(const h3_block_config* cfg, int32_t n_blocks, const h3_block_weights* w,
                            const h3_packed_meta* meta, const void* x_in, void* x_out, void* workspace,
                            size_t ws_bytes, cudaStream_t stream) {
  if (!w) return H3_ERR_NULL;
  if (n_blocks < 1) return H3_ERR_SHAPE;
  for (int b = 0; b < n_blocks; ++b) {
    h3_status s = check_block_args(cfg, &w[b], meta, x_in, x_out, workspace, ws_bytes);
    if (s != H3_OK) return s;
  }
  if (ws_bytes < chain_ws_bytes(*cfg, n_blocks, meta->n_rows, meta->n_timesteps)) return H3_ERR_WORKSPACE;
  return chain_impl(cfg, n_blocks, w, meta, x_in, x_out, workspace, ws_bytes, stream);
}

// ===========================================================================
// the chain as one CUDA graph
// ===========================================================================
struct h3_graph {
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t exec = nullptr;
};

h3_status h3_blocks_graph_create(const h3_block_config* cfg, int32_t n_blocks, const h3_block_weights* w,
                                 const h3_packed_meta* meta, const void* x_in, void* x_out, void* workspace,
                                 size_t ws_bytes, h3_graph** out) {
  if (!out) return H3_ERR_NULL;
  *out = nullptr;
  if (!w) return H3_ERR_NULL;
  if (n_blocks < 1) return H3_ERR_SHAPE;
  for (int b = 0; b < n_blocks; ++b) {
    h3_status s = check_block_args(cfg, &w[b], meta, x_in, x_out, workspace, ws_bytes);
    if (s != H3_OK) return s;
  }
  if (ws_bytes < chain_ws_bytes(*cfg, n_blocks, meta->n_rows, meta->n_timesteps)) return H3_ERR_WORKSPACE;
  cudaStream_t cap = nullptr;
  if (cudaStreamCreateWithFlags(&cap, cudaStreamNonBlocking) != cudaSuccess) return H3_ERR_CUDA;
  h3_status s = H3_OK;
  if (cudaStreamBeginCapture(cap, cudaStreamCaptureModeThreadLocal) != cudaSuccess) {
    cudaStreamDestroy(cap);
    return H3_ERR_CUDA;
  }
  s = chain_impl(cfg, n_blocks, w, meta, x_in, x_out, workspace, ws_bytes, cap);
  cudaGraph_t g = nullptr;
  const cudaError_t e_end = cudaStreamEndCapture(cap, &g);
  cudaStreamDestroy(cap);
  if (s != H3_OK || e_end != cudaSuccess || !g) {
    if (g) cudaGraphDestroy(g);
    cudaGetLastError();
    return s != H3_OK ? s : H3_ERR_CUDA;
  }
  cudaGraphExec_t ex = nullptr;
  if (cudaGraphInstantiate(&ex, g, 0) != cudaSuccess) {
    cudaGraphDestroy(g);
    cudaGetLastError();
    return H3_ERR_CUDA;
  }
  h3_graph* hg = new (std::nothrow) h3_graph;
  if (!hg) {
    cudaGraphExecDestroy(ex);
    cudaGraphDestroy(g);
    return H3_ERR_CUDA;
  }
  hg->graph = g;
  hg->exec = ex;
  *out = hg;
  set_kernel_info("blocks graph: %d blocks captured (side-stream fork/join and programmatic launches as edges)",
                  n_blocks);
  return H3_OK;
}

h3_status h3_graph_launch(h3_graph* g, cudaStream_t stream) {
  if (!g || !g->exec) return H3_ERR_NULL;
  return cudaGraphLaunch(g->exec, stream) == cudaSuccess ? H3_OK : H3_ERR_CUDA;
}

h3_status h3_graph_destroy(h3_graph* g) {
  if (!g) return H3_ERR_NULL;
  if (g->exec) cudaGraphExecDestroy(g->exec);
  if (g->graph) cudaGraphDestroy(g->graph);
  delete g;
  return H3_OK;
}

// ===========================================================================
// token refiner: the block's stages with the identity AdaLN table and
// text / timestep-0 / zero-position metadata written into the workspace
// ===========================================================================
namespace {
size_t refiner_meta_bytes(int64_t S) { return al256((size_t)5 * (size_t)S * 4); }

h3_status check_refiner_weights(const h3_block_weights* w) {
  if (!w) return H3_ERR_NULL;
  const void* req[] = {w->norm1_g, w->norm2_g, w->w_qkv, w->q_norm_g, w->k_norm_g, w->w_o, w->w_fc1, w->w_fc2};
  for (const void* p : req) {
    if (!p) return H3_ERR_NULL;
    if (!al16(p)) return H3_ERR_ALIGN;
  }
  const void* opt[] = {w->b_qkv, w->b_o, w->b_fc1, w->b_fc2};
  for (const void* p : opt)
    if (!al16n(p)) return H3_ERR_ALIGN;
  return H3_OK;
}
}  // namespace

size_t h3_refiner_workspace_bytes(const h3_block_config* cfg, int32_t n_rows) {
  if (check_cfg(cfg) != H3_OK || n_rows < 1) return 0;
  return ws_layout(*cfg, n_rows, 1).total + refiner_meta_bytes(n_rows);
}

h3_status h3_refiner_forward(const h3_block_config* cfg, int32_t n_blocks, const h3_block_weights* w,
                             const void* final_norm_g, int32_t n_rows, const void* x_in, void* x_out,
                             void* workspace, size_t ws_bytes, cudaStream_t stream) {
  h3_status s = check_cfg(cfg);
  if (s != H3_OK) return s;
  if (n_rows < 1 || n_blocks < 0 || (n_blocks == 0 && !final_norm_g)) return H3_ERR_SHAPE;
  if (n_blocks > 0 && !w) return H3_ERR_NULL;
  for (int b = 0; b < n_blocks; ++b)
    if ((s = check_refiner_weights(&w[b])) != H3_OK) return s;
  if (!x_in || !x_out || !workspace) return H3_ERR_NULL;
  if (!al16(x_in) || !al16(x_out) || !al16n(final_norm_g) || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return H3_ERR_ALIGN;
  const WsLayout L = ws_layout(*cfg, n_rows, 1);
  if (ws_bytes < L.total + refiner_meta_bytes(n_rows)) return H3_ERR_WORKSPACE;
  uint8_t* base = static_cast<uint8_t*>(workspace);
  void* table = base + L.table;
  void* h = base + L.h;
  void* qkv = base + L.qkv;
  void* o = base + L.o;
  void* x1 = base + L.x1;
  SkScratch sk{reinterpret_cast<float*>(base + L.sk_part), reinterpret_cast<uint32_t*>(base + L.sk_flags), 0};
  int32_t* tag = reinterpret_cast<int32_t*>(base + L.total);
  int32_t* tidx = tag + n_rows;
  int32_t* pos = tidx + n_rows;
  const int S = n_rows, I = cfg->n_heads * 128;
  if ((s = cuda_st(launch_refiner_setup(S, cfg->dim, static_cast<__nv_bfloat16*>(table), tag, tidx, pos, sk.flags,
                                        (int)gemm_sk_flag_words(), stream))) != H3_OK)
    return s;
  const h3_packed_meta m{S, 1, tag, tidx, pos, nullptr};
  for (int b = 0; b < n_blocks; ++b) {
    const void* xi = b == 0 ? x_in : x_out;
    const h3_block_weights& wb = w[b];
    const __nv_bfloat16* q = static_cast<const __nv_bfloat16*>(qkv);
    if ((s = run_modulate(*cfg, m, table, 0, xi, wb.norm1_g, h, stream)) != H3_OK) return s;
    if ((s = run_qkv(*cfg, m, h, wb.w_qkv, wb.b_qkv, wb.q_norm_g, wb.k_norm_g, qkv, stream)) != H3_OK) return s;
    if ((s = run_attention(S, cfg->n_heads, q, q + 128, q + 256, 3 * I, 384, o, nullptr, stream)) != H3_OK)
      return s;
    if ((s = run_resid_gemm(*cfg, m, table, 2, o, I, wb.w_o, wb.b_o, xi, x1, stream, &sk)) != H3_OK) return s;
    if ((s = run_modulate(*cfg, m, table, 1, x1, wb.norm2_g, h, stream)) != H3_OK) return s;
    if ((s = run_ffn_up(*cfg, S, h, wb.w_fc1, wb.b_fc1, qkv, stream)) != H3_OK) return s;
    if ((s = run_resid_gemm(*cfg, m, table, 5, qkv, cfg->ffn_dim, wb.w_fc2, wb.b_fc2, x1, x_out, stream, &sk)) !=
        H3_OK)
      return s;
  }
  if (final_norm_g)   // row-local, so in place on x_out
    if ((s = run_modulate(*cfg, m, table, 0, n_blocks > 0 ? x_out : x_in, final_norm_g, x_out, stream)) != H3_OK)
      return s;
  return H3_OK;
}

size_t h3_adaln_table_workspace_bytes(const h3_block_config* cfg) {
  if (check_cfg(cfg) != H3_OK) return 0;
  return adaln_scratch_bytes(*cfg);
}

h3_status h3_adaln_table(const h3_block_config* cfg, const void* w_ada, const void* b_ada, const float* t_cond,
                         int32_t n_timesteps, void* table_out, void* workspace, size_t ws_bytes,
                         cudaStream_t stream) {
  h3_status s = check_cfg(cfg);
  if (s != H3_OK) return s;
  if (!w_ada || !t_cond || !table_out || !workspace) return H3_ERR_NULL;
  if (n_timesteps < 1 || n_timesteps > 16) return H3_ERR_UNSUPPORTED;
  if (!al16(w_ada) || !al16n(b_ada) || !al16(table_out) || (reinterpret_cast<uintptr_t>(t_cond) & 3u) ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return H3_ERR_ALIGN;
  if (ws_bytes < adaln_scratch_bytes(*cfg)) return H3_ERR_WORKSPACE;
  return run_adaln_table(*cfg, w_ada, b_ada, t_cond, n_timesteps, table_out, workspace, stream);
}

h3_status h3_adaln_table_noalloc(const h3_block_config* cfg, const void* w_ada, const void* b_ada,
                                 const float* t_cond, int32_t n_timesteps, void* table_out, cudaStream_t stream) {
  h3_status s = check_cfg(cfg);
  if (s != H3_OK) return s;
  if (cfg->cond_dim > kNoAllocMaxCond) return H3_ERR_UNSUPPORTED;
  if (!w_ada || !t_cond || !table_out) return H3_ERR_NULL;
  if (n_timesteps < 1 || n_timesteps > kAdalnRows) return H3_ERR_UNSUPPORTED;
  if (!al16(w_ada) || !al16n(b_ada) || !al16(table_out) || (reinterpret_cast<uintptr_t>(t_cond) & 3u))
    return H3_ERR_ALIGN;
  void* u = nullptr;
  if ((s = noalloc_scratch(&u)) != H3_OK) return s;
  // the SiLU kernel rewrites every row of the scratch (zeros beyond T), so no
  // contents of an earlier call are read
  return run_adaln_table(*cfg, w_ada, b_ada, t_cond, n_timesteps, table_out, u, stream);
}

h3_status h3_adaln_modulate(const h3_block_config* cfg, const h3_packed_meta* meta, const void* table,
                            int32_t branch, const void* x, const void* norm_g, void* h_out, cudaStream_t stream) {
  h3_status s = check_cfg(cfg);
  if (s != H3_OK) return s;
  if (!meta) return H3_ERR_NULL;
  if (meta->n_rows < 1) return H3_ERR_SHAPE;
  if (!meta->token_tag || !meta->timestep_index) return H3_ERR_NULL;
  if (meta->n_timesteps < 1 || meta->n_timesteps > 16) return H3_ERR_UNSUPPORTED;
  if (branch != 0 && branch != 1) return H3_ERR_SHAPE;
  if (!table || !x || !norm_g || !h_out) return H3_ERR_NULL;
  if (!al16(table) || !al16(x) || !al16(norm_g) || !al16(h_out)) return H3_ERR_ALIGN;
  return run_modulate(*cfg, *meta, table, branch, x, norm_g, h_out, stream);
}

h3_status h3_qkv_projection(const h3_block_config* cfg, const h3_packed_meta* meta, const void* h,
                            const void* w_qkv, const void* b_qkv, const void* q_norm_g, const void* k_norm_g,
                            void* qkv_out, cudaStream_t stream) {
  h3_status s = check_cfg(cfg);
  if (s != H3_OK) return s;
  if ((s = check_meta(meta, false)) != H3_OK) return s;
  if (!h || !w_qkv || !q_norm_g || !k_norm_g || !qkv_out) return H3_ERR_NULL;
  if (!al16(h) || !al16(w_qkv) || !al16n(b_qkv) || !al16(q_norm_g) || !al16(k_norm_g) || !al16(qkv_out))
    return H3_ERR_ALIGN;
  return run_qkv(*cfg, *meta, h, w_qkv, b_qkv, q_norm_g, k_norm_g, qkv_out, stream);
}

h3_status h3_rope_qknorm(const h3_block_config* cfg, int32_t n_rows, const int32_t* pos_thw, void* q, void* k,
                         int64_t row_stride_elems, int64_t head_stride_elems, const void* q_norm_g,
                         const void* k_norm_g, cudaStream_t stream) {
  h3_status s = check_cfg(cfg);
  if (s != H3_OK) return s;
  if (n_rows < 1) return H3_ERR_SHAPE;
  if (!pos_thw || !q || !k || !q_norm_g || !k_norm_g) return H3_ERR_NULL;
  if (row_stride_elems < 128 || head_stride_elems < 128) return H3_ERR_SHAPE;
  if ((row_stride_elems & 7) || (head_stride_elems & 7)) return H3_ERR_ALIGN;
  if (!al16(q) || !al16(k) || !al16(q_norm_g) || !al16(k_norm_g)) return H3_ERR_ALIGN;
  RopeArgs a{};
  a.S = n_rows;
  a.H = cfg->n_heads;
  a.q = static_cast<__nv_bfloat16*>(q);
  a.k = static_cast<__nv_bfloat16*>(k);
  a.row_stride = row_stride_elems;
  a.head_stride = head_stride_elems;
  a.q_gain = static_cast<const __nv_bfloat16*>(q_norm_g);
  a.k_gain = static_cast<const __nv_bfloat16*>(k_norm_g);
  a.pos = pos_thw;
  a.eps = cfg->eps;
  fill_omega(a.omega, cfg->rope_theta);
  a.qk_elems = (size_t)(n_rows - 1) * (size_t)row_stride_elems + (size_t)(a.H - 1) * (size_t)head_stride_elems + 128;
  a.err = device_error_word();
  CUtensorMap tq, tk;
  const uint32_t hb = (uint32_t)rope_qknorm_heads_per_unit(a.H);
  if (!make_tmap_rope(&tq, q, (uint64_t)n_rows, (uint64_t)a.H, (uint64_t)row_stride_elems,
                      (uint64_t)head_stride_elems, hb) ||
      !make_tmap_rope(&tk, k, (uint64_t)n_rows, (uint64_t)a.H, (uint64_t)row_stride_elems,
                      (uint64_t)head_stride_elems, hb))
    return H3_ERR_CUDA;
  return cuda_st(launch_rope_qknorm(tq, tk, a, num_sms(), stream));
}

h3_status h3_attention(int32_t n_rows, int32_t n_heads, const void* q, const void* k, const void* v,
                       int64_t row_stride_elems, int64_t head_stride_elems, void* o, float* lse_opt,
                       cudaStream_t stream) {
  if (n_rows < 1 || n_heads < 1 || n_heads > 65535) return H3_ERR_SHAPE;
  if (!q || !k || !v || !o) return H3_ERR_NULL;
  if (row_stride_elems < 128 || head_stride_elems < 128) return H3_ERR_SHAPE;
  if ((row_stride_elems & 7) || (head_stride_elems & 7)) return H3_ERR_ALIGN;
  if (!al16(q) || !al16(k) || !al16(v) || !al16(o) || (reinterpret_cast<uintptr_t>(lse_opt) & 3u))
    return H3_ERR_ALIGN;
  return run_attention(n_rows, n_heads, q, k, v, row_stride_elems, head_stride_elems, o, lse_opt, stream);
}

h3_status h3_out_projection(const h3_block_config* cfg, const h3_packed_meta* meta, const void* table,
                            const void* o, const void* w_o, const void* b_o, const void* x, void* x_out,
                            cudaStream_t stream) {
  h3_status s = check_cfg(cfg);
  if (s != H3_OK) return s;
  if (!meta) return H3_ERR_NULL;
  if (meta->n_rows < 1) return H3_ERR_SHAPE;
  if (!meta->token_tag || !meta->timestep_index) return H3_ERR_NULL;
  if (meta->n_timesteps < 1 || meta->n_timesteps > 16) return H3_ERR_UNSUPPORTED;
  if (!table || !o || !w_o || !x || !x_out) return H3_ERR_NULL;
  if (!al16(table) || !al16(o) || !al16(w_o) || !al16n(b_o) || !al16(x) || !al16(x_out)) return H3_ERR_ALIGN;
  return run_resid_gemm(*cfg, *meta, table, 2, o, cfg->n_heads * 128, w_o, b_o, x, x_out, stream);
}

h3_status h3_ffn_up_swiglu(const h3_block_config* cfg, int32_t n_rows, const void* h, const void* w_fc1,
                           const void* b_fc1, void* a_out, cudaStream_t stream) {
  h3_status s = check_cfg(cfg);
  if (s != H3_OK) return s;
  if (n_rows < 1) return H3_ERR_SHAPE;
  if (!h || !w_fc1 || !a_out) return H3_ERR_NULL;
  if (!al16(h) || !al16(w_fc1) || !al16n(b_fc1) || !al16(a_out)) return H3_ERR_ALIGN;
  return run_ffn_up(*cfg, n_rows, h, w_fc1, b_fc1, a_out, stream);
}

h3_status h3_ffn_down_residual(const h3_block_config* cfg, const h3_packed_meta* meta, const void* table,
                               const void* a, const void* w_fc2, const void* b_fc2, const void* x1, void* y_out,
                               cudaStream_t stream) {
  h3_status s = check_cfg(cfg);
  if (s != H3_OK) return s;
  if (!meta) return H3_ERR_NULL;
  if (meta->n_rows < 1) return H3_ERR_SHAPE;
  if (!meta->token_tag || !meta->timestep_index) return H3_ERR_NULL;
  if (meta->n_timesteps < 1 || meta->n_timesteps > 16) return H3_ERR_UNSUPPORTED;
  if (!table || !a || !w_fc2 || !x1 || !y_out) return H3_ERR_NULL;
  if (!al16(table) || !al16(a) || !al16(w_fc2) || !al16n(b_fc2) || !al16(x1) || !al16(y_out)) return H3_ERR_ALIGN;
  return run_resid_gemm(*cfg, *meta, table, 5, a, cfg->ffn_dim, w_fc2, b_fc2, x1, y_out, stream);
}

h3_status h3_linear(int32_t M, int32_t N, int32_t K, const void* x, const void* w, const void* b, void* y,
                    cudaStream_t stream) {
  if (M < 1 || N < 1 || K < 64) return H3_ERR_SHAPE;
  if (K % 64 || N % 8) return H3_ERR_UNSUPPORTED;
  if (!x || !w || !y) return H3_ERR_NULL;
  if (!al16(x) || !al16(w) || !al16n(b) || !al16(y)) return H3_ERR_ALIGN;
  const GemmPlan pl = gemm_plan(EPI_PLAIN, M, N, 0, 0);
  CUtensorMap tA, tB;
  if (!make_tmap_2d(&tA, x, M, K, K, 128) || !make_tmap_2d(&tB, w, N, K, K, (uint32_t)pl.b_rows))
    return H3_ERR_CUDA;
  GemmArgs a{};
  gemm_common(a, M, K, pl.num_n);
  gemm_set_plan(a, pl);
  a.out = static_cast<__nv_bfloat16*>(y);
  a.ldo = N;
  a.bias = static_cast<const __nv_bfloat16*>(b);
  a.n_valid = N;
  return cuda_st(launch_gemm(EPI_PLAIN, pl.bn, tA, tB, a, stream));
}

// ===========================================================================
// input side
// ===========================================================================
namespace {
h3_status patch_common(int32_t C, int32_t T, int32_t H, int32_t W, const float* a, const float* b) {
  if (C < 1 || T < 1 || H < 2 || W < 2 || (H & 1) || (W & 1)) return H3_ERR_SHAPE;
  if ((long long)C * T * H * W > (1LL << 40)) return H3_ERR_SHAPE;
  if (!a || !b) return H3_ERR_NULL;
  return H3_OK;
}
}  // namespace

h3_status h3_patch_pack(int32_t C, int32_t T, int32_t H, int32_t W, const float* latent, float* rows,
                        cudaStream_t stream) {
  h3_status s = patch_common(C, T, H, W, latent, rows);
  if (s != H3_OK) return s;
  return cuda_st(launch_patch_pack(C, T, H, W, latent, rows, false, stream));
}

h3_status h3_patch_unpack(int32_t C, int32_t T, int32_t H, int32_t W, const float* rows, float* latent,
                          cudaStream_t stream) {
  h3_status s = patch_common(C, T, H, W, rows, latent);
  if (s != H3_OK) return s;
  return cuda_st(launch_patch_pack(C, T, H, W, rows, latent, true, stream));
}

h3_status h3_input_projection(const h3_block_config* cfg, int32_t n, int32_t K, const float* src, const float* w,
                              const float* b, const int32_t* dst_rows, int32_t n_rows, void* x_out,
                              cudaStream_t stream) {
  h3_status s = check_cfg(cfg);
  if (s != H3_OK) return s;
  if (n < 0 || n_rows < 1) return H3_ERR_SHAPE;
  if (K < 4 || K > kInputProjMaxK || (K & 3)) return H3_ERR_UNSUPPORTED;
  if (n == 0) return H3_OK;
  if (!src || !w || !dst_rows || !x_out) return H3_ERR_NULL;
  if (!al16(src) || !al16(w) || !al16(x_out)) return H3_ERR_ALIGN;
  InputProjArgs a{};
  a.n = n;
  a.K = K;
  a.D = cfg->dim;
  a.n_dst = n_rows;
  a.src = src;
  a.w = w;
  a.b = b;
  a.dst = dst_rows;
  a.out = static_cast<__nv_bfloat16*>(x_out);
  a.err = device_error_word();
  return cuda_st(launch_input_proj(a, stream));
}

h3_status h3_packed_index_copy(const h3_block_config* cfg, int32_t n, const void* src, const int32_t* dst_rows,
                               int32_t n_rows, void* x_out, cudaStream_t stream) {
  h3_status s = check_cfg(cfg);
  if (s != H3_OK) return s;
  if (n < 0 || n_rows < 1) return H3_ERR_SHAPE;
  if (n == 0) return H3_OK;
  if (!src || !dst_rows || !x_out) return H3_ERR_NULL;
  if (!al16(src) || !al16(x_out)) return H3_ERR_ALIGN;
  return cuda_st(launch_index_copy(n, cfg->dim, static_cast<const __nv_bfloat16*>(src), dst_rows, n_rows,
                                   static_cast<__nv_bfloat16*>(x_out), device_error_word(), stream));
}

h3_status h3_timestep_embedding(const h3_block_config* cfg, int32_t n_timesteps, const float* t, const float* w1,
                                const float* b1, const float* w2, const float* b2, float* scratch, float* t_cond,
                                cudaStream_t stream) {
  h3_status s = check_cfg(cfg);
  if (s != H3_OK) return s;
  if (n_timesteps < 1 || n_timesteps > 16) return H3_ERR_UNSUPPORTED;
  if (!t || !w1 || !w2 || !scratch || !t_cond) return H3_ERR_NULL;
  if (!al16(w1) || !al16(w2) || !al16(scratch) || !al16(t_cond) || !al16n(b1) || !al16n(b2)) return H3_ERR_ALIGN;
  const int T = n_timesteps, D = cfg->dim, C = cfg->cond_dim;
  float* e = scratch;                 // [T][256]
  float* h = scratch + (size_t)T * 256;   // [T][D]
  if ((s = cuda_st(launch_sinusoid(T, t, e, stream))) != H3_OK) return s;
  if ((s = cuda_st(launch_rows_linear(T, 256, D, e, w1, b1, 1, h, stream))) != H3_OK) return s;
  return cuda_st(launch_rows_linear(T, D, C, h, w2, b2, 0, t_cond, stream));
}

// ===========================================================================
// output side and sampler
// ===========================================================================
h3_status h3_sigma_schedule(int32_t n_points, float shift, float* sigmas, int32_t* n_sigmas, cudaStream_t stream) {
  if (!sigmas || !n_sigmas) return H3_ERR_NULL;
  if (n_points < 2 || n_points > (1 << 20) || !std::isfinite(shift) || !(shift > 0.0f)) return H3_ERR_SHAPE;
  return cuda_st(launch_sigma_grid(n_points, shift, sigmas, n_sigmas, stream));
}

h3_status h3_ode_step(int64_t n, const float* xt, const float* v, float sigma, float sigma_next, float* x_next,
                      cudaStream_t stream) {
  if (n < 0) return H3_ERR_SHAPE;
  if (!std::isfinite(sigma) || !(sigma > 0.0f) || !std::isfinite(sigma_next) || sigma_next < 0.0f)
    return H3_ERR_SHAPE;
  if (n == 0) return H3_OK;
  if (!xt || !v || !x_next) return H3_ERR_NULL;
  if (!al16(xt) || !al16(v) || !al16(x_next)) return H3_ERR_ALIGN;
  return cuda_st(launch_ode_step((long long)n, xt, v, sigma, sigma_next, x_next, stream));
}

h3_status h3_noise_mix(int64_t n, const float* x0, const float* noise, float t, float* out, cudaStream_t stream) {
  if (n < 0 || !std::isfinite(t) || t < 0.0f || t > 1.0f) return H3_ERR_SHAPE;
  if (n == 0) return H3_OK;
  if (!x0 || !noise || !out) return H3_ERR_NULL;
  if (!al16(x0) || !al16(noise) || !al16(out)) return H3_ERR_ALIGN;
  return cuda_st(launch_noise_mix((long long)n, x0, noise, t, out, stream));
}

h3_status h3_select_rows(int32_t n_rows, const int32_t* token_tag, int32_t tag, int32_t* rows, int32_t* n_selected,
                         cudaStream_t stream) {
  if (n_rows < 0) return H3_ERR_SHAPE;
  if (!token_tag || !rows || !n_selected) return H3_ERR_NULL;
  return cuda_st(launch_select_rows(n_rows, token_tag, tag, rows, n_selected, stream));
}

h3_status h3_final_adaln_tables(const h3_block_config* cfg, int32_t n_tables, const float* const* w_fin,
                                const float* const* b_fin, const float* t_cond, int32_t n_timesteps,
                                float* const* tables, cudaStream_t stream) {
  h3_status s = check_cfg(cfg);
  if (s != H3_OK) return s;
  if (n_tables < 1 || n_tables > kFinalAdalnMaxTables || n_timesteps < 1 || n_timesteps > 16)
    return H3_ERR_UNSUPPORTED;
  if (!w_fin || !tables || !t_cond) return H3_ERR_NULL;
  if (!al16(t_cond)) return H3_ERR_ALIGN;
  FinalAdalnArgs a{};
  a.n_tables = n_tables;
  for (int m = 0; m < n_tables; ++m) {
    if (!w_fin[m] || !tables[m]) return H3_ERR_NULL;
    const float* bm = b_fin ? b_fin[m] : nullptr;
    if (!al16(w_fin[m]) || !al16n(bm) || !al16(tables[m])) return H3_ERR_ALIGN;
    a.w[m] = w_fin[m];
    a.b[m] = bm;
    a.out[m] = tables[m];
  }
  a.t_cond = t_cond;
  a.T = n_timesteps;
  a.C = cfg->cond_dim;
  a.rows = 2 * cfg->dim;
  return cuda_st(launch_final_adaln(a, stream));
}

h3_status h3_final_adaln_table(const h3_block_config* cfg, const float* w_fin, const float* b_fin,
                               const float* t_cond, int32_t n_timesteps, float* table, cudaStream_t stream) {
  return h3_final_adaln_tables(cfg, 1, &w_fin, &b_fin, t_cond, n_timesteps, &table, stream);
}

h3_status h3_output_head(const h3_block_config* cfg, int32_t n_rows, int32_t n_sel, const int32_t* rows,
                         const int32_t* timestep_index, int32_t n_timesteps, const void* x, const float* table,
                         const float* w_head, const float* b_head, int32_t P, float* v_out, cudaStream_t stream) {
  h3_status s = check_cfg(cfg);
  if (s != H3_OK) return s;
  if (n_rows < 1 || n_sel < 0 || n_sel > n_rows) return H3_ERR_SHAPE;
  if (P < 1 || P > kOutputHeadMaxP || n_timesteps < 1 || n_timesteps > 16) return H3_ERR_UNSUPPORTED;
  if (!rows || !timestep_index || !x || !table || !w_head || !v_out) return H3_ERR_NULL;
  if (!al16(x) || !al16(table) || !al16(w_head)) return H3_ERR_ALIGN;
  if (n_sel == 0) return H3_OK;
  OutputHeadArgs a{};
  a.n_sel = n_sel;
  a.S = n_rows;
  a.T = n_timesteps;
  a.D = cfg->dim;
  a.P = P;
  a.rows = rows;
  a.tidx = timestep_index;
  a.x = static_cast<const __nv_bfloat16*>(x);
  a.table = table;
  a.w = w_head;
  a.b = b_head;
  a.out = v_out;
  a.eps = cfg->eps;
  a.err = device_error_word();
  return cuda_st(launch_output_head(a, stream));
}

h3_status h3_sync_check(cudaStream_t stream, int32_t timeout_ms) {
  cudaEvent_t ev;
  if (cudaEventCreateWithFlags(&ev, cudaEventDisableTiming) != cudaSuccess) return H3_ERR_CUDA;
  if (cudaEventRecord(ev, stream) != cudaSuccess) {
    cudaEventDestroy(ev);
    return H3_ERR_CUDA;
  }
  const auto t0 = std::chrono::steady_clock::now();
  cudaError_t e;
  while ((e = cudaEventQuery(ev)) == cudaErrorNotReady) {
    const auto ms =
        std::chrono::duration_cast<std::chrono::milliseconds>(std::chrono::steady_clock::now() - t0).count();
    if (ms > timeout_ms) {
      cudaEventDestroy(ev);
      return H3_ERR_TIMEOUT;
    }
    std::this_thread::sleep_for(std::chrono::microseconds(50));
  }
  cudaEventDestroy(ev);
  if (e != cudaSuccess) return H3_ERR_CUDA;
  uint32_t* p = device_error_word();
  if (!p) return H3_ERR_CUDA;
  uint32_t words[2] = {0u, 0u};
  if (cudaMemcpy(words, p, sizeof(words), cudaMemcpyDeviceToHost) != cudaSuccess) return H3_ERR_CUDA;
  const uint32_t bits = words[0];
  if (bits || words[1]) {
    if (cudaMemset(p, 0, sizeof(words)) != cudaSuccess) return H3_ERR_CUDA;
    if (cudaDeviceSynchronize() != cudaSuccess) return H3_ERR_CUDA;
  }
  if (bits & DEVERR_TIMEOUT) {
    note_error_site(words[1]);
    return H3_ERR_TIMEOUT;
  }
  if (bits & DEVERR_BOUNDS) {
    note_error_site(words[1]);
    return H3_ERR_BOUNDS;
  }
  if (bits & DEVERR_INDEX) return H3_ERR_INDEX;
  return H3_OK;
}

const char* h3_status_string(h3_status s) {
  switch (s) {
    case H3_OK: return "ok";
    case H3_ERR_NULL: return "null pointer argument";
    case H3_ERR_SHAPE: return "size out of range";
    case H3_ERR_ALIGN: return "pointer or stride not 16-byte aligned";
    case H3_ERR_UNSUPPORTED: return "unsupported configuration (fails closed)";
    case H3_ERR_INDEX: return "device saw a bad tag, timestep index or position";
    case H3_ERR_CUDA: return "CUDA runtime error";
    case H3_ERR_TIMEOUT: return "device wait or stream synchronisation timed out";
    case H3_ERR_WORKSPACE: return "workspace too small";
    case H3_ERR_BOUNDS: return "bounds-checked build: a kernel access fell outside its buffer";
  }
  return "unknown status";
}

h3_status h3_last_error_site(char* buf, size_t len) {
  if (!buf || len == 0) return H3_ERR_NULL;
  std::lock_guard<std::mutex> lk(g_site_mu);
  snprintf(buf, len, "%s", g_site);
  return H3_OK;
}

h3_status h3_last_kernel_info(char* buf, size_t len) {
  if (!buf || len == 0) return H3_ERR_NULL;
  snprintf(buf, len, "%s", g_info);
  return H3_OK;
}

const char* h3_version(void) { return "libh3 0.1 sm_103a tcgen05"; }

}  // extern "C"
