/*
 * libh3 -- MiniMax-H3 Omni-Transformer block forward on one GB300 (sm_103a).
 *
 * The operations are defined by the RL-Kernel RFC "[MiniMax-H3][CUDA/ROCm]
 * WS1/WS2 kernel roadmap, ablation matrix and integration plan" ("the RFC"):
 * section 2 (Omni-Transformer and mixed-precision fingerprint tables),
 * section 3 (figure 2, one H3 block), section 4 (the H3-specific arithmetic
 * rules) and the work items of section 5.  The checkpoint layout of the QKV
 * rows follows the "h3-metal" README, section "Checkpoint layout and media
 * pipeline".
 *
 * Conventions shared by every entry point:
 *   - All tensor pointers are DEVICE pointers owned by the caller.  The
 *     library never allocates or frees device memory; where scratch space is
 *     needed the caller passes a workspace sized by the matching *_bytes call.
 *   - bf16 tensors are row-major, 16-byte aligned, with every row stride a
 *     multiple of 16 bytes.  Weights are [out][in].
 *   - Calls are stream-ordered and asynchronous.  Argument errors are returned
 *     synchronously, before anything is launched, and nothing is launched
 *     then.  Unsupported geometry fails closed (H3_ERR_UNSUPPORTED); there is
 *     no fallback path.
 *   - Bad metadata values found on the device (a tag outside {0,1,2}, a
 *     timestep index outside [0,T), a position outside [0, 2^24)) do not
 *     fault: the kernel records the error in a device error word, leaves the
 *     row's output unwritten and carries on.  h3_sync_check reads and clears
 *     that word.  A device-side wait that exceeds its time limit (2 s) is
 *     recorded the same way (H3_ERR_TIMEOUT), together with the site of the
 *     first such wait (h3_last_error_site).  The timeout bit is sticky: until
 *     h3_sync_check clears it, every library kernel whose CTAs start after
 *     it is recorded skips its work (it reads the bit in its prologue), so
 *     one lost signal ends the whole queue of work within about one time
 *     limit instead of costing one limit per later launch.  Results of calls
 *     made in that window are undefined; the status says so.
 *   - Results are deterministic: a given call on a given GPU gives bitwise
 *     the same output every time.  With H3_GEMM_SK=0 in the environment every
 *     reduction has a fixed order that does not depend on the row count, the
 *     launch geometry or the SM count (RFC section 4, numerical contract
 *     items 1-3).  By default the block's O and FC2 projections run
 *     stream-K where whole tiles would leave SM pairs idle: their fp32 partial
 *     sums over k-ranges are added in k order, with split points fixed by the
 *     row-tile count and the resident SM-pair count (recorded in
 *     h3_last_kernel_info as stream-k=<pairs>).  For long documents only the
 *     tiles of the last waves are split that way; the others run whole
 *     (sk-whole-tiles=<tiles> in the same record).
 */
#ifndef H3_H_
#define H3_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  H3_OK = 0,
  H3_ERR_NULL = 1,         /* a required pointer is NULL */
  H3_ERR_SHAPE = 2,        /* a size is out of range (e.g. n_rows < 1) */
  H3_ERR_ALIGN = 3,        /* a pointer or stride breaks the 16-byte rule */
  H3_ERR_UNSUPPORTED = 4,  /* a configuration this library does not implement */
  H3_ERR_INDEX = 5,        /* the device saw a bad tag / timestep index / position */
  H3_ERR_CUDA = 6,         /* a CUDA runtime call failed */
  H3_ERR_TIMEOUT = 7,      /* a device-side wait or h3_sync_check timed out */
  H3_ERR_WORKSPACE = 8,    /* the workspace is smaller than required */
  H3_ERR_BOUNDS = 9        /* bounds-checked build only: a kernel's global access fell outside the
                              buffer its call's arguments describe (skipped; h3_last_error_site) */
} h3_status;

/* Block widths (RFC s2, "Omni-Transformer fingerprint").  Supported:
 * head_dim == 128, rope_freqs_per_axis == 16, rope_channels == 96,
 * dim, cond_dim multiples of 64 (cond_dim <= 2816), ffn_dim a multiple of
 * 128, n_heads in [1, 1024].  H3 itself: dim 5376, n_heads 56, ffn_dim 14336,
 * cond_dim 2688, eps 1e-5, rope_theta 10000. */
typedef struct {
  int32_t dim;                  /* D, residual width */
  int32_t n_heads;              /* H */
  int32_t head_dim;             /* 128 */
  int32_t ffn_dim;              /* F, SwiGLU hidden width */
  int32_t cond_dim;             /* C, timestep embedding width into the AdaLN projection */
  int32_t rope_freqs_per_axis;  /* 16 */
  int32_t rope_channels;        /* 96 */
  float eps;                    /* RMSNorm epsilon (block and Q/K norms) */
  float rope_theta;             /* 10000 */
} h3_block_config;

/* One block's weights, all bf16 device pointers.  Biases may be NULL.
 *   w_ada  [18*D][C], b_ada [18*D]: AdaLN projection.  Output channel
 *          n = m*6*D + c*D + d is (modality m, chunk c, channel d), chunks
 *          in the order shift_msa, scale_msa, gate_msa, shift_mlp, scale_mlp,
 *          gate_mlp.
 *   norm1_g, norm2_g [D]: block RMSNorm gains.
 *   w_qkv  [H*3*128][D], b_qkv [H*3*128]: rows interleaved per head,
 *          head h owning rows h*384 .. h*384+383 as q(128), k(128), v(128).
 *   q_norm_g, k_norm_g [128]: per-head Q/K RMSNorm gains, shared by heads.
 *   w_o    [D][H*128], b_o [D]
 *   w_fc1  [2F][D], b_fc1 [2F]: rows 0..F-1 gate (SiLU'd), F..2F-1 value.
 *   w_fc2  [D][F], b_fc2 [D]                                               */
typedef struct {
  const void *w_ada, *b_ada;
  const void *norm1_g, *norm2_g;
  const void *w_qkv, *b_qkv;
  const void *q_norm_g, *k_norm_g;
  const void *w_o, *b_o;
  const void *w_fc1, *b_fc1;
  const void *w_fc2, *b_fc2;
} h3_block_weights;

/* Packed-row metadata of one document (RFC s3: the row identity tuple; s4:
 * the index tensors, tags and positions carry meaning and are inputs of the
 * arithmetic, not incidental metadata).  Device pointers:
 *   token_tag [S] int32 in {0 video, 1 text, 2 audio}
 *   timestep_index [S] int32 in [0, T)
 *   pos_thw [S][3] int32 (t, h, w) in [0, 2^24)
 *   t_cond [T][C] fp32, the timestep embedding before the AdaLN SiLU.       */
typedef struct {
  int32_t n_rows;        /* S >= 1 */
  int32_t n_timesteps;   /* T in [1, 16] */
  const int32_t *token_tag;
  const int32_t *timestep_index;
  const int32_t *pos_thw;
  const float *t_cond;
} h3_packed_meta;

/* ----------------------------------------------------------------------- */
/* The block                                                                */
/* ----------------------------------------------------------------------- */

/* Bytes of workspace h3_block_forward / h3_blocks_forward need for S rows and
 * T timestep rows.  Returns 0 for an invalid configuration. */
size_t h3_block_workspace_bytes(const h3_block_config *cfg, int32_t n_rows, int32_t n_timesteps);

/* One Omni-Transformer block forward (RFC s3 figure 2; s5 work items
 * adaln_projection_3mod through h3_ffn_down_gemm, composed as in
 * ws1_one_h3_block):
 *   table = bf16(SiLU(t_cond) W_ada^T + b_ada)            as [3T][6][D]
 *   r     = timestep_index*3 + token_tag
 *   h1    = bf16(rms(x) g1 (1 + scale_msa[r]) + shift_msa[r])
 *   qkv   = bf16(h1 W_qkv^T + b_qkv);  q,k <- RoPE(bf16(rms_128(.) g))
 *   o     = bf16(softmax(q k^T / sqrt(128)) v)             (no mask)
 *   x1    = bf16(x + gate_msa[r] bf16(o W_o^T + b_o))
 *   h2    = bf16(rms(x1) g2 (1 + scale_mlp[r]) + shift_mlp[r])
 *   a     = bf16(SiLU(g) u),  [g | u] = bf16(h2 W_fc1^T + b_fc1)
 *   y     = bf16(x1 + gate_mlp[r] bf16(a W_fc2^T + b_fc2))
 * x_in, x_out: bf16 [S][D]; x_out may alias x_in.  The workspace (device,
 * 256-byte aligned, >= h3_block_workspace_bytes) is scratch: its contents on
 * return are the block's intermediates (layout not part of the ABI).
 * When D is a multiple of 128, the AdaLN chunks that norm1 does not read are
 * computed on a stream the library owns (one per device), overlapping the
 * QKV projection; the caller's stream waits for them before the O
 * projection, so the work stays ordered on the caller's stream.
 * Reduction order: when whole 256-column tiles would leave SM pairs idle
 * (a few hundred rows), the O and FC2 projections share each tile's K range
 * out over several SM pairs and add the fp32 partial sums in k order
 * (stream-K).  The split is fixed for a given row count and GPU, so repeated
 * calls are bitwise equal, but it changes with the row count and the number
 * of SMs; set H3_GEMM_SK=0 in the environment for one fixed MMA sequence per
 * output element at every size (the RFC's strict order, section 4). */
h3_status h3_block_forward(const h3_block_config *cfg, const h3_block_weights *w,
                           const h3_packed_meta *meta, const void *x_in, void *x_out,
                           void *workspace, size_t ws_bytes, cudaStream_t stream);

/* h3_block_forward from and to host memory, for callers whose activations
 * live on the host: copies x_host (bf16 [S][D]) and the packed metadata that
 * meta_host points to (token_tag, timestep_index, pos_thw, t_cond: host
 * arrays of the sizes h3_packed_meta states) into staging space at the end
 * of the workspace with one cudaMemcpyAsync each, runs the block there, and
 * copies the result to y_host (bf16 [S][D]); x_host and y_host may be the
 * same buffer.  The copy of x_host runs on a stream the library owns (one
 * per device), after the caller's earlier work on `stream`, so that it
 * overlaps the AdaLN table; the block waits for it before reading x.  Everything is ordered on `stream` and the call returns before
 * the copies complete: synchronize the stream before reading y_host or
 * reusing the inputs.  Host buffers should be page-locked (cudaHostAlloc or
 * pinned), otherwise the copies are synchronous.  The weights stay device
 * pointers.  Workspace: device, 256-byte aligned, at least
 * h3_block_host_workspace_bytes (the block workspace plus the staging). */
size_t h3_block_host_workspace_bytes(const h3_block_config *cfg, int32_t n_rows, int32_t n_timesteps);
h3_status h3_block_forward_host(const h3_block_config *cfg, const h3_block_weights *w,
                                const h3_packed_meta *meta_host, const void *x_host, void *y_host,
                                void *workspace, size_t ws_bytes, cudaStream_t stream);
/* The same for the chain w[0 .. n_blocks) of h3_blocks_forward: one copy in,
 * the blocks in order on the device, one copy out.  Workspace: at least
 * h3_blocks_host_workspace_bytes (the chain workspace plus the staging). */
size_t h3_blocks_host_workspace_bytes(const h3_block_config *cfg, int32_t n_blocks, int32_t n_rows,
                                      int32_t n_timesteps);
h3_status h3_blocks_forward_host(const h3_block_config *cfg, int32_t n_blocks, const h3_block_weights *w,
                                 const h3_packed_meta *meta_host, const void *x_host, void *y_host,
                                 void *workspace, size_t ws_bytes, cudaStream_t stream);

/* As h3_block_forward, recording cudaEvent_t events[k] on the stream after
 * launch stage k, for k = 0..min(n_events, 8)-1, stages in order: 0 AdaLN
 * table (the chunks on the caller's stream), 1 norm1/modulate, 2 QKV +
 * QK-norm + RoPE, 3 attention, 4 O projection + gated residual,
 * 5 norm2/modulate, 6 FC1 + SwiGLU, 7 FC2 + gated residual.  When the AdaLN
 * chunks 2-5 run on the library's side stream, events[8] and events[9] (if
 * n_events > 9) are recorded on that stream before and after them.  events
 * may be NULL (then identical to h3_block_forward). */
h3_status h3_block_forward_profiled(const h3_block_config *cfg, const h3_block_weights *w,
                                    const h3_packed_meta *meta, const void *x_in, void *x_out,
                                    void *workspace, size_t ws_bytes, cudaStream_t stream,
                                    void *const *events, int32_t n_events);

/* How h3_block_forward schedules the AdaLN table for this config and row
 * count on the current device: the number of SMs given to the chunks 2-5 on
 * the library's side stream, or 0 when the whole table runs on the caller's
 * stream.  A scheduling detail (no counterpart on the pages); results are
 * identical either way. */
int32_t h3_block_adaln_side_ctas(const h3_block_config *cfg, int32_t n_rows);

/* How many kernels one h3_blocks_forward call of n_blocks blocks over n_rows
 * rows launches on the current device (h3_block_forward: n_blocks = 1); 0
 * for invalid arguments.  Per block: the SiLU rows and the AdaLN table (two
 * launches when split over the side stream), norm1, QKV, attention, O,
 * norm2 (not launched when H3_NORM_FUSE=1 in the environment lets an O
 * projection that runs stream-K carry it in its epilogue), FC1, FC2; a chain that computes its tables up front
 * launches the SiLU rows once and one table kernel per 64 blocks instead.
 * A scheduling detail (no counterpart on the pages). */
int32_t h3_blocks_kernel_count(const h3_block_config *cfg, int32_t n_blocks, int32_t n_rows);

/* A chain of n_blocks blocks (RFC s2 fingerprint row "Transformer layers"; s5
 * ws1_full_h3_transformer, without the refiner and heads): block b reads the
 * output of block b-1 and uses weights w[b] (a HOST array of n_blocks
 * structs of device pointers).  x_out may alias x_in.  Where a single block
 * would get no overlap for its AdaLN table (h3_block_adaln_side_ctas is 0,
 * as for long documents), the chain computes the tables of all its blocks up
 * front: one SiLU launch and one table launch per 64 blocks, streaming every
 * block's AdaLN weights once, and each block then starts at norm1.  The
 * tables are the same numbers either way.  Workspace: device, 256-byte
 * aligned, at least h3_blocks_workspace_bytes (the block workspace, plus the
 * chain's tables when it computes them up front); H3_ERR_WORKSPACE below. */
size_t h3_blocks_workspace_bytes(const h3_block_config *cfg, int32_t n_blocks, int32_t n_rows,
                                 int32_t n_timesteps);
h3_status h3_blocks_forward(const h3_block_config *cfg, int32_t n_blocks,
                            const h3_block_weights *w, const h3_packed_meta *meta,
                            const void *x_in, void *x_out, void *workspace, size_t ws_bytes,
                            cudaStream_t stream);

/* The same chain captured once into a CUDA graph and replayed with one launch
 * (one graph per denoiser evaluation).  h3_blocks_graph_create
 * records the launches h3_blocks_forward would make for these arguments
 * (pointers and sizes are baked in; the buffers' contents are read at each
 * replay) and instantiates the graph; h3_graph_launch replays it on a
 * stream; h3_graph_destroy frees it.  The block's side-stream fork and join
 * and the programmatic dependent launches become edges of the graph.
 * Validation errors as for h3_blocks_forward; H3_ERR_CUDA if capture or
 * instantiation fails.  *graph is NULL on error. */
typedef struct h3_graph h3_graph;
h3_status h3_blocks_graph_create(const h3_block_config *cfg, int32_t n_blocks,
                                 const h3_block_weights *weights, const h3_packed_meta *meta,
                                 const void *x_in, void *x_out, void *workspace,
                                 size_t workspace_bytes, h3_graph **graph);
h3_status h3_graph_launch(h3_graph *graph, cudaStream_t stream);
h3_status h3_graph_destroy(h3_graph *graph);

/* ----------------------------------------------------------------------- */
/* Stages (each is one kernel launch)                                       */
/* ----------------------------------------------------------------------- */

/* AdaLN modulation table (RFC s5 adaln_projection_3mod; s4: the SiLU runs at
 * the timestep-embedding precision and only its result is cast to bf16):
 * table[t][n] = bf16(sum_k bf16(SiLU(t_cond[t][k])) w_ada[n][k] + b_ada[n])
 * for n < 18*D, stored [T][18*D] bf16 (= [3T][6][D]).  t_cond fp32 [T][C]
 * with 1 <= T <= 16.  b_ada may be NULL.  workspace: device scratch of at
 * least h3_adaln_table_workspace_bytes bytes, 256-byte aligned (holds the
 * bf16 SiLU rows). */
size_t h3_adaln_table_workspace_bytes(const h3_block_config *cfg);
h3_status h3_adaln_table(const h3_block_config *cfg, const void *w_ada, const void *b_ada,
                         const float *t_cond, int32_t n_timesteps, void *table_out,
                         void *workspace, size_t ws_bytes, cudaStream_t stream);

/* The AdaLN table of h3_adaln_table without any caller-provided scratch.
 * The pages have no counterpart: this entry point exists for callers that
 * cannot allocate device memory themselves (code handed only its input and
 * output buffers by a host framework that owns the allocator, or a
 * latency-critical loop that must not call cudaMalloc, which can synchronise
 * the device).  Same arguments and result as h3_adaln_table, minus the
 * workspace.  The scratch is a file-scope device array of 16 x 2816 bf16
 * (90,112 bytes) that every GPU loading the library holds until exit; configs
 * with cond_dim > 2816 or n_timesteps > 16 are rejected (H3_ERR_UNSUPPORTED).
 * The first call on a device looks up the array's device address with that
 * device current; make that first call before any stream capture.  Each
 * GPU has its own copy of the array, and on one GPU every call shares it:
 * calls that can overlap on the GPU (for example on two streams with no
 * ordering between them) race, so serialise them.  Each call keeps its
 * contents until the next; nothing has to be cleared first, because a call
 * rewrites every scratch row it reads (rows past n_timesteps with zeros).
 * Allocates nothing. */
h3_status h3_adaln_table_noalloc(const h3_block_config *cfg, const void *w_ada, const void *b_ada,
                                 const float *t_cond, int32_t n_timesteps, void *table_out,
                                 cudaStream_t stream);

/* RMSNorm + AdaLN modulation of one branch (RFC s2 fingerprint row "Block
 * norm", eps 1e-5; s5 h3_rmsnorm and adaln_row_gather):
 *   h[i] = bf16(x[i] / sqrt(mean(x[i]^2) + eps) * g * (1 + scale[r_i]) + shift[r_i])
 * with r_i = timestep_index[i]*3 + token_tag[i], shift/scale the chunks of
 * branch 0 (attention: shift_msa, scale_msa) or 1 (MLP: shift_mlp,
 * scale_mlp) of table [3T][6][D].  x, h_out bf16 [S][D]; norm_g bf16 [D]. */
h3_status h3_adaln_modulate(const h3_block_config *cfg, const h3_packed_meta *meta,
                            const void *table, int32_t branch, const void *x, const void *norm_g,
                            void *h_out, cudaStream_t stream);

/* QKV projection with the per-head Q/K RMSNorm and MM-RoPE in its epilogue
 * (RFC s5 h3_qkv_gemm, h3_qk_rmsnorm_d128, h3_mm_rope_3axis_partial; s4: the
 * Q/K norm precedes RoPE, whose frequencies are built in FP32 and which
 * rotates 96 channels and no more).  h bf16 [S][D]; qkv_out bf16
 * [S][H][3][128]: q and k slots hold the normed, rotated values, the v slot
 * bf16(h W_v^T + b_v).  RoPE as in h3_rope_qknorm. */
h3_status h3_qkv_projection(const h3_block_config *cfg, const h3_packed_meta *meta,
                            const void *h, const void *w_qkv, const void *b_qkv,
                            const void *q_norm_g, const void *k_norm_g, void *qkv_out,
                            cudaStream_t stream);

/* Standalone per-head Q/K RMSNorm + partial three-axis MM-RoPE, in place
 * (RFC s2 rows "Q/K preprocessing", "Position encoding", "RoPE frequencies",
 * "Rotary channels").  For every row i and head h, on the 128 channels at
 *   q + i*row_stride + h*head_stride   (and the same for k):
 *   n_j = bf16(x_j / sqrt(mean(x^2) + eps) * g_j)
 *   for j < 48, with band a = j/16 (t, h, w) and f = j%16:
 *     theta = fp32(pos_thw[i][a]) * fp32(rope_theta^(-f/16))    (fp32)
 *     out_j    = bf16(n_j cos(theta) - n_{j+48} sin(theta))
 *     out_j+48 = bf16(n_{j+48} cos(theta) + n_j sin(theta))
 *   out_j = n_j for j in [96, 128).
 * Strides are in elements, multiples of 8.  q and k bf16. */
h3_status h3_rope_qknorm(const h3_block_config *cfg, int32_t n_rows, const int32_t *pos_thw,
                         void *q, void *k, int64_t row_stride_elems, int64_t head_stride_elems,
                         const void *q_norm_g, const void *k_norm_g, cudaStream_t stream);

/* Full non-causal, unmasked multi-head attention over one packed document
 * (RFC s2 fingerprint row "Attention"; s4: no causal, padding or
 * per-modality mask in the released path; s5 h3_full_attention):  o[i][h*128 + c] = bf16(sum_j P_ij v[j][h][c]) with
 * P = softmax_j(q_i . k_j / sqrt(128)) in fp32.  q, k, v bf16, element
 * (row i, head h, channel c) at ptr + i*row_stride + h*head_stride + c
 * (strides in elements, multiples of 8).  o bf16 [S][H*128].  lse_opt: NULL
 * or fp32 [H][S] receiving log(sum_j exp(q_i.k_j/sqrt(128))). */
h3_status h3_attention(int32_t n_rows, int32_t n_heads, const void *q, const void *k,
                       const void *v, int64_t row_stride_elems, int64_t head_stride_elems,
                       void *o, float *lse_opt, cudaStream_t stream);

/* Output projection + gated residual of the attention branch (RFC s5
 * h3_attention_o_gemm and adaln_gate_residual; s4: residual plus the row's
 * gate times the sublayer output, in that order):  x_out = bf16(x + gate_msa[r] bf16(o W_o^T + b_o)).
 * o bf16 [S][H*128]; x, x_out bf16 [S][D] (may alias); table [3T][6][D]. */
h3_status h3_out_projection(const h3_block_config *cfg, const h3_packed_meta *meta,
                            const void *table, const void *o, const void *w_o, const void *b_o,
                            const void *x, void *x_out, cudaStream_t stream);

/* FC1 with SwiGLU in its epilogue (RFC s5 h3_ffn_gate_up_gemm and h3_swiglu):
 * a = bf16(SiLU(g) u) in fp32, [g | u] = bf16(h W_fc1^T + b_fc1).
 * h bf16 [S][D]; a_out bf16 [S][F]. */
h3_status h3_ffn_up_swiglu(const h3_block_config *cfg, int32_t n_rows, const void *h,
                           const void *w_fc1, const void *b_fc1, void *a_out,
                           cudaStream_t stream);

/* FC2 + gated residual of the MLP branch (RFC s5 h3_ffn_down_gemm and
 * adaln_gate_residual): y = bf16(x1 + gate_mlp[r] bf16(a W_fc2^T + b_fc2)).
 * a bf16 [S][F]; x1, y_out bf16 [S][D] (may alias). */
h3_status h3_ffn_down_residual(const h3_block_config *cfg, const h3_packed_meta *meta,
                               const void *table, const void *a, const void *w_fc2,
                               const void *b_fc2, const void *x1, void *y_out,
                               cudaStream_t stream);

/* Plain bf16 projection y = bf16(x W^T + b) with fp32 accumulation (a BF16
 * module of the RFC s2 mixed-precision table, with its output cast).  x [M][K], W [N][K],
 * y [M][N]; K a multiple of 64, N a multiple of 8; b may be NULL. */
h3_status h3_linear(int32_t M, int32_t N, int32_t K, const void *x, const void *w,
                    const void *b, void *y, cudaStream_t stream);

/* ----------------------------------------------------------------------- */
/* Input side of one denoiser evaluation                                   */
/* ----------------------------------------------------------------------- */

/* Video latent to patch rows (RFC s2: visual VAE latent of C = 24 channels,
 * transformer video patch (1, 2, 2), flattened width 96; s5
 * video_patch_pack_unpack).  latent fp32 [C][T][H][W] (one batch row), rows
 * fp32 [T*(H/2)*(W/2)][4C]: row (t, h/2, w/2) with t slowest (the order of the
 * video positions), feature (c, dh, dw) with c slowest.  H and W even; both
 * device pointers.  h3_patch_unpack is the exact inverse. */
h3_status h3_patch_pack(int32_t C, int32_t T, int32_t H, int32_t W, const float *latent, float *rows,
                        cudaStream_t stream);
h3_status h3_patch_unpack(int32_t C, int32_t T, int32_t H, int32_t W, const float *rows, float *latent,
                          cudaStream_t stream);

/* FP32 input projection of one modality (RFC s5
 * video_input_projection_fp32 96 -> 5376, audio_input_projection_fp32
 * 32 -> 5376): x_out[dst_rows[i]] = bf16(src[i] W^T + b), fp32 inputs,
 * weights and accumulation, one rounding to bf16 (the h3-metal README's patch
 * projection), written straight into the packed residual stream.  src fp32
 * [n][K], w fp32 [D][K], b fp32 [D] or NULL, dst_rows int32 [n] (device),
 * x_out bf16 [n_rows][D]; K a multiple of 4, 4 <= K <= 128; D = cfg->dim.  A
 * destination outside [0, n_rows) is reported (H3_ERR_INDEX) and skipped. */
h3_status h3_input_projection(const h3_block_config *cfg, int32_t n, int32_t K, const float *src,
                              const float *w, const float *b, const int32_t *dst_rows, int32_t n_rows,
                              void *x_out, cudaStream_t stream);

/* Row scatter into the packed stream (RFC s5 packed_index_copy):
 * x_out[dst_rows[i]] = src[i] for bf16 rows of D = cfg->dim (e.g. the refined
 * text rows).  Zero-initialising the stream first is the caller's memset;
 * rows no modality writes stay zero.  Bad destinations are reported and
 * skipped. */
h3_status h3_packed_index_copy(const h3_block_config *cfg, int32_t n, const void *src, const int32_t *dst_rows,
                               int32_t n_rows, void *x_out, cudaStream_t stream);

/* Timestep conditioning rows (RFC s2: sinusoid width 256, timestep MLP
 * 256 -> 5376 -> 2688, FP32; s5 timestep_sinusoid_h3, timestep_mlp_fp32):
 * e = [cos(t f_i) | sin(t f_i)], f_i = exp(-ln(10000) i / 128), i < 128, with
 * t = 1 - sigma as given (no 0..1000 scaling); h = SiLU(e W1^T + b1);
 * t_cond = h W2^T + b2.  t fp32 [T]; w1 fp32 [D][256]; w2 fp32 [C][D]; b1, b2
 * or NULL; scratch fp32 [T][256 + D]; t_cond fp32 [T][C]; 1 <= T <= 16,
 * D = cfg->dim, C = cfg->cond_dim.  All device pointers. */
h3_status h3_timestep_embedding(const h3_block_config *cfg, int32_t n_timesteps, const float *t,
                                const float *w1, const float *b1, const float *w2, const float *b2,
                                float *scratch, float *t_cond, cudaStream_t stream);

/* ----------------------------------------------------------------------- */
/* Token refiner                                                            */
/* ----------------------------------------------------------------------- */

/* Workspace for h3_refiner_forward over n_rows rows (0 when cfg is unsupported). */
size_t h3_refiner_workspace_bytes(const h3_block_config *cfg, int32_t n_rows);

/* Token refiner over the projected text rows (RFC s2: "Text projection
 * 5120 -> 5376, then 2-layer token refiner"; s5 token_refiner_block: pre-norm
 * attention/FFN blocks without AdaLN or RoPE; the ledger's refiner ends with
 * a final RMSNorm).  Each of the n_blocks blocks is the Omni-Transformer block
 * with the modulation removed: h1 = bf16(rms(x) g1), per-head Q/K RMSNorm,
 * full unmasked attention over the n_rows rows, x1 = bf16(x + bf16(o W_o^T +
 * b_o)), h2 = bf16(rms(x1) g2), SwiGLU FFN, y = bf16(x1 + bf16(a W_fc2^T +
 * b_fc2)); then, when final_norm_g is not NULL, x_out = bf16(rms(y) g_final).
 * weights: array of n_blocks (w_ada and b_ada are not used); final_norm_g bf16
 * [D] or NULL; x_in, x_out bf16 [n_rows][D] (may alias).  It runs the block's
 * kernels with an identity modulation table (shift 0, scale 0, gate 1) and
 * zero positions, written into the workspace. */
h3_status h3_refiner_forward(const h3_block_config *cfg, int32_t n_blocks, const h3_block_weights *weights,
                             const void *final_norm_g, int32_t n_rows, const void *x_in, void *x_out,
                             void *workspace, size_t workspace_bytes, cudaStream_t stream);

/* ----------------------------------------------------------------------- */
/* Output side and sampler of one denoiser evaluation                      */
/* ----------------------------------------------------------------------- */

/* Sigma grid of one modality's scheduler (RFC s2 "Scheduler fingerprint":
 * sigma transform s*sigma/(1+(s-1)*sigma), grid = shifted linspace(1, 0,
 * n_points) with consecutive fp32 duplicates removed; s5 h3_sigma_schedule).
 * Point i is the fp64 value 1 - i/(n_points-1) rounded to fp32, shifted in
 * fp32 with one rounding per operation (num = s*sigma, den = 1 + (s-1)*sigma,
 * num/den); a terminal zero is appended and consecutive equal values
 * collapsed (the linspace's own zero and the terminal zero become one), so
 * the grid holds n_points values and n_points - 1 model evaluations.  The
 * video scheduler uses shift 12, the audio one 3.  sigmas: device float
 * [n_points + 1] (the first *n_sigmas used); n_sigmas: device int32.  Both are
 * written by the device (read them after the stream).  Errors:
 * n_points < 2 or > 1048576, shift not finite or <= 0 -> H3_ERR_SHAPE;
 * NULL -> H3_ERR_NULL. */
h3_status h3_sigma_schedule(int32_t n_points, float shift, float *sigmas, int32_t *n_sigmas,
                            cudaStream_t stream);

/* One Euler step of the data-ward flow (RFC s2 "Velocity convention" x0 = xt +
 * sigma*v and "Euler update" x_next = r*xt + (1-r)*x0 with r =
 * sigma_next/sigma; s5 h3_ode_step): fp32, one rounding per operation in that
 * order, no fused multiply-add, so the result is bit-reproducible.  xt, v,
 * x_next: device float [n], 16-byte aligned; x_next may alias xt.  sigma must
 * be finite and > 0, sigma_next finite and >= 0 (H3_ERR_SHAPE otherwise);
 * n = 0 does nothing. */
h3_status h3_ode_step(int64_t n, const float *xt, const float *v, float sigma, float sigma_next,
                      float *x_next, cudaStream_t stream);

/* Conditioning-anchor noise mix out = t*x0 + (1-t)*noise (RFC s5
 * conditioning_noise_mix), fp32 as written.  All arrays device float [n],
 * 16-byte aligned; out may alias either input.  t finite in [0, 1]. */
h3_status h3_noise_mix(int64_t n, const float *x0, const float *noise, float t, float *out,
                       cudaStream_t stream);

/* Rows of one modality in packed order (RFC s5 packed_index_select): rows
 * receives the indices i < n_rows with token_tag[i] == tag, ascending, and
 * n_selected their count (both device memory, written by the device).
 * token_tag and rows: device int32 [n_rows]. */
h3_status h3_select_rows(int32_t n_rows, const int32_t *token_tag, int32_t tag, int32_t *rows,
                         int32_t *n_selected, cudaStream_t stream);

/* Final AdaLN table of one modality (RFC s5 final_adaln_out; the ledger's
 * "H3 final layer"): table[t][0][:] = shift, table[t][1][:] = scale, from
 * SiLU(t_cond[t]) W_fin^T + b_fin in fp32 (an FP32 module of the RFC s2
 * mixed-precision table).  w_fin fp32 [2D][C] (rows 0..D-1 shift, D..2D-1
 * scale), b_fin fp32 [2D] or NULL, t_cond fp32 [T][C], table fp32 [T][2][D];
 * D = cfg->dim, C = cfg->cond_dim, 1 <= T <= 16.  All device pointers. */
h3_status h3_final_adaln_table(const h3_block_config *cfg, const float *w_fin, const float *b_fin,
                               const float *t_cond, int32_t n_timesteps, float *table,
                               cudaStream_t stream);

/* The final AdaLN tables of up to four modalities in one launch, their
 * weights streamed back to back (the video and audio tables of an
 * evaluation).  Table m is exactly what h3_final_adaln_table gives for
 * w_fin[m], b_fin[m] and tables[m], bit for bit.  w_fin, b_fin and tables are
 * HOST arrays of n_tables device pointers; b_fin may be NULL (no bias for
 * any table) or hold NULL entries.  1 <= n_tables <= 4, else
 * H3_ERR_UNSUPPORTED; a NULL weight or table pointer gives H3_ERR_NULL. */
h3_status h3_final_adaln_tables(const h3_block_config *cfg, int32_t n_tables, const float *const *w_fin,
                                const float *const *b_fin, const float *t_cond, int32_t n_timesteps,
                                float *const *tables, cudaStream_t stream);

/* Velocity head of one modality (RFC s5 video_output_projection_fp32 5376 ->
 * 96, audio_output_projection_fp32 5376 -> 32): for i < n_sel and r = rows[i],
 *   m = RMSNorm(x[r]) * (1 + table[tidx[r]][1]) + table[tidx[r]][0]
 * (plain RMSNorm, no gain, eps cfg->eps, fp32), then v_out[i] = m W_head^T +
 * b_head in fp32.  x bf16 [n_rows][D]; rows device int32 [n_sel] (e.g. from
 * h3_select_rows); timestep_index device int32 [n_rows]; table fp32 [T][2][D];
 * w_head fp32 [P][D]; b_head fp32 [P] or NULL; v_out fp32 [n_sel][P];
 * 1 <= P <= 128.  A row index or timestep index out of range is reported
 * through the device error word (h3_sync_check -> H3_ERR_INDEX) and its
 * output row left unwritten. */
h3_status h3_output_head(const h3_block_config *cfg, int32_t n_rows, int32_t n_sel,
                         const int32_t *rows, const int32_t *timestep_index, int32_t n_timesteps,
                         const void *x, const float *table, const float *w_head, const float *b_head,
                         int32_t P, float *v_out, cudaStream_t stream);

/* ----------------------------------------------------------------------- */
/* Status, errors, provenance                                               */
/* ----------------------------------------------------------------------- */

/* Waits for the stream's work (polling, at most timeout_ms; never blocks
 * forever), then reads and clears the device error word.  Returns H3_OK,
 * H3_ERR_INDEX (bad metadata was seen), H3_ERR_TIMEOUT (a device wait gave up,
 * or the stream did not finish within timeout_ms) or H3_ERR_CUDA. */
h3_status h3_sync_check(cudaStream_t stream, int32_t timeout_ms);

const char *h3_status_string(h3_status s);

/* Provenance of the most recent launch from this host thread (RFC s4 item 10,
 * s5 h3_operator_trace): kernel id, tile shape, pipeline depth, accumulator
 * type, grid.  Writes a NUL-terminated string of at most len bytes. */
h3_status h3_last_kernel_info(char *buf, size_t len);

/* Where the first device-side wait that ran out was, as recorded on the
 * device and read by the most recent h3_sync_check of this process that
 * returned H3_ERR_TIMEOUT: "none", or the kernel ("gemm", "attention-1q",
 * "attention-2q", "adaln-table", "rope-qknorm") and the wait (an mbarrier at
 * a shared-memory byte offset, or a stream-K partial-sum flag).  Diagnostic
 * only: the pages define no counterpart.  Writes a NUL-terminated string of
 * at most len bytes; H3_ERR_NULL when buf is NULL or len is 0. */
h3_status h3_last_error_site(char *buf, size_t len);

/* Library version string. */
const char *h3_version(void);

#ifdef __cplusplus
}
#endif
#endif /* H3_H_ */
