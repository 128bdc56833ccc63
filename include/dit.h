/*
 * dit.h -- C ABI of the GB300 (sm_103a) library for one FLUX.2 [klein]-style DiT
 * denoising step.
 *
 * What the step computes (sources, by page title and section):
 *   - "flux2-klein-p100a" model card, task table: 4 steps, guidance 1.0, no CFG, so each
 *     step is one DiT call; Caveats: all 512 padded text rows enter the DiT with no mask,
 *     text features are encoder layers 9, 18, 27 concatenated to [512, 7680], and the
 *     modulation is global per step, not per block.
 *   - "tt_flux2_klein -- Python reference", Modules: tt_dit.py runs 5 dual-stream and
 *     20 single-stream blocks; host.py builds the token ids and RoPE; "Things that are
 *     easy to get wrong": RoPE is 32 dims per axis at theta 2000 on adjacent pairs, and
 *     reference image i gets t = 10 + 10*i.
 *   The pages do not write the block maths out; the readings this library implements
 *   (LayerNorm eps 1e-6, (1 + scale) LN(x) + shift, raw gates, per-head QK-RMSNorm
 *   before RoPE, SwiGLU with the gate first, no biases, sinusoidal timestep embedding of
 *   1000*sigma) are stated beside each entry point.
 *
 * Conventions for every entry point:
 *   - Pointers marked "dev" are caller-owned device memory, 16-byte aligned; "host" ones
 *     are host memory.  The library never allocates device memory in these calls and
 *     never frees caller memory.  Weights stay owned by the caller; the structs below
 *     hold pointers only.
 *   - Tensors are bf16 (raw 16-bit storage) unless stated; row-major; "[A, B]" lists the
 *     outermost dimension first.
 *   - Device work is enqueued asynchronously on `stream` (NULL = the legacy default
 *     stream).  A return value reports what was known at launch time only.
 *   - Every argument is validated before anything is launched.  An invalid argument
 *     returns DIT_ERR_INVALID_ARG, an unsupported configuration DIT_ERR_UNSUPPORTED, a
 *     too-small workspace DIT_ERR_WORKSPACE; in those cases nothing is launched and no
 *     memory is touched.  A failed launch returns DIT_ERR_CUDA.
 *   - Kernels never trap or spin forever: a device-side wait that runs past its limit
 *     writes a status word in the workspace and the kernel unwinds; dit_sync_status()
 *     reports it as DIT_ERR_TIMEOUT.
 *   - No C++ exception crosses this boundary.  Calls on different workspaces and
 *     streams may run concurrently from different host threads, with two exceptions,
 *     both process-wide state: the timing functions (dit_timing_*), and
 *     dit_modulation_static, whose calls all share one fixed device array (two of its
 *     calls that overlap on the GPU race on it).
 */
#ifndef DIT_H_
#define DIT_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same handle as cudaStream_t. */
typedef struct CUstream_st* dit_stream_t;

typedef enum {
  DIT_OK = 0,
  DIT_ERR_INVALID_ARG = 1,
  DIT_ERR_UNSUPPORTED = 2,
  DIT_ERR_WORKSPACE = 3,
  DIT_ERR_CUDA = 4,
  DIT_ERR_TIMEOUT = 5
} dit_status;

/* Model widths.  Supported: head_dim == 128, hidden == heads * 128 with hidden / 256 in
 * {1, 2, 3, 4, 5, 6, 8, 10, 12, 14, 16} (hidden <= 4096), mlp_hidden % 128 == 0 and
 * <= 2^19, in_channels % 32 == 0 and <= 2^20, txt_dim % 8 == 0 and <= 2^20, axes_dim[i]
 * even with sum == head_dim, rope_theta > 0, eps > 0.
 * klein 4B: {3072, 24, 128, 9216, 5, 20, 128, 7680, 2000.f, {32,32,32,32}, 1e-6f}. */
typedef struct {
  int hidden, heads, head_dim, mlp_hidden, n_dual, n_single, in_channels, txt_dim;
  float rope_theta;
  int axes_dim[4];
  float eps;
} dit_config;

/* Joint sequence of one step: per batch row, rows [text | target image | references];
 * N = n_txt + n_img + n_ref.  n_txt >= 1, n_img >= 1, n_ref >= 0, 1 <= batch <= 64. */
typedef struct {
  int batch, n_txt, n_img, n_ref;
} dit_shape;

/* Timestep MLP and the global modulation projection: t_in [H, 256], t_out [H, H],
 * mod [17H, H]. */
typedef struct {
  const void *t_in, *t_out, *mod;
} dit_mod_weights;

/* One stream of a dual-stream block: qkv [3H, H] (rows q | k | v), q_norm [128],
 * k_norm [128], out [H, H], mlp_in [2F, H] in the PACKED layout of dit_pack_mlp_in,
 * mlp_out [H, F].  No biases. */
typedef struct {
  const void *qkv, *q_norm, *k_norm, *out, *mlp_in, *mlp_out;
} dit_stream_weights;

typedef struct {
  dit_stream_weights img, txt;
} dit_dual_weights;

/* A single-stream block: qkv_mlp [3H + 2F, H] whose first 3H rows are q | k | v and
 * whose last 2F rows are the MLP-in in the PACKED layout of dit_pack_mlp_in;
 * q_norm [128], k_norm [128]; out [H, H + F] over the concatenation [attn | act]. */
typedef struct {
  const void *qkv_mlp, *q_norm, *k_norm, *out;
} dit_single_weights;

/* Low-precision (e4m3) copy of one projection matrix W [rows, cols]: q [rows, cols] e4m3
 * bytes in the same row order as W and scale [rows] fp32, one per output row, with
 * W ~= scale[n] * q[n, :] (from dit_quantize_rows_fp8).  q == NULL means "this projection
 * stays bf16".  The "dit_prec" precision knob of the "tt_flux2_klein -- Python reference"
 * KleinTT constructor names a precision choice for the projections without fixing a format;
 * e4m3 with per-row scales is this library's reading of it. */
typedef struct {
  const void* q;
  const float* scale;
} dit_fp8_matrix;

/* e4m3 copies of a single-stream block's projections: the fused QKV + MLP-in [3H + 2F, H]
 * (packed row order of qkv_mlp; both pointers required) and, optionally, the
 * out-projection [H, H + F] (out.q NULL: bf16). */
typedef struct {
  const void* qkv_mlp_q;
  const float* qkv_mlp_scale;
  dit_fp8_matrix out;
} dit_single_fp8;

/* e4m3 copies of one stream's projections in a dual-stream block: qkv [3H, H], mlp_in
 * [2F, H] (packed row order), out [H, H], mlp_out [H, F].  Each projection runs in e4m3
 * when BOTH streams give its copy and in bf16 when neither does (the two streams share one
 * launch); one stream alone is an argument error. */
typedef struct {
  dit_fp8_matrix qkv, mlp_in, out, mlp_out;
} dit_stream_fp8;
typedef struct {
  dit_stream_fp8 img, txt;
} dit_dual_fp8;

/* All weights.  `dual` and `single` are HOST arrays of n_dual and n_single entries
 * (they hold device pointers); they must stay valid for the duration of each call.
 * x_emb [H, in_channels], ctx_emb [H, txt_dim], proj_out [in_channels, H].
 * single_fp8 / dual_fp8: NULL for the bf16 path; else HOST arrays of n_single / n_dual
 * entries naming e4m3 copies of the block projections.  An e4m3 projection takes its input
 * quantised per token row (scale = max|row| / 448): the modulated activations by the adaLN
 * kernel, the attention output and the SwiGLU activations by a quantising pass before the
 * out-projections; the product is accumulated in fp32 and dequantised in the GEMM epilogue
 * before RMSNorm / RoPE / SwiGLU / the gated residual.  Attention, norms, modulation,
 * embedders and the final projection stay bf16. */
typedef struct {
  dit_config cfg;
  dit_mod_weights mod;
  const void *x_emb, *ctx_emb, *proj_out;
  const dit_dual_weights* dual;
  const dit_single_weights* single;
  const dit_single_fp8* single_fp8;
  const dit_dual_fp8* dual_fp8;
} dit_weights;

/* Human-readable name of a status code (static string, never NULL). */
const char* dit_status_string(dit_status s);

/* Fill *cfg with the klein 4B widths listed above. */
dit_status dit_config_klein(dit_config* cfg);

/* Bytes of workspace that every *_fwd / dit_modulation / dit_attention call on this
 * config and shape needs (the largest of them; dit_step_host included).  The workspace
 * is caller-owned device memory; its first 256 bytes hold the device status word and
 * must be zeroed once by the caller before first use (the library clears it again in
 * dit_sync_status). */
dit_status dit_workspace_size(const dit_config* cfg, const dit_shape* shape, size_t* bytes);

/* Host maths: the (t, h, w, l) position id of every row of the joint sequence, written
 * to ids_host [N, 4] int32.  Text row i: (0, 0, 0, i), padded rows continuing the
 * count; target token (r, c) of the grid_h x grid_w patch grid, row-major: (0, r, c, 0);
 * reference i (ref_grids_host[2i] rows x ref_grids_host[2i+1] cols, row-major):
 * (10 + 10*i, r, c, 0) ("tt_flux2_klein -- Python reference", "Things that are easy to
 * get wrong", and Modules: host.py).  Requires grid_h * grid_w == shape->n_img and the
 * reference grids to sum to shape->n_ref.  Runs on the host; touches no device. */
dit_status dit_token_ids(const dit_shape* shape, int grid_h, int grid_w, const int* ref_grids_host, int n_refs,
                         int32_t* ids_host);

/* RoPE table of a sequence: for every row and every adjacent pair p of the 128-dim head
 * (axis a owns dims [sum(axes_dim[<a]), +axes_dim[a]); its pair j turns by
 * pos_a * theta^(-2j / axes_dim[a])), table_dev[(row * 64 + p) * 2 + {0, 1}] =
 * {cos, sin} as fp32, angles evaluated in fp64 ("tt_flux2_klein -- Python reference",
 * "Things that are easy to get wrong").  ids_dev [n, 4] int32 device, table_dev
 * [n, 64, 2] fp32 device.  Build it once per shape; every block call reads it. */
dit_status dit_rope_table(const dit_config* cfg, const int32_t* ids_dev, int n, float* table_dev,
                          dit_stream_t stream);

/* Weight preparation: rearrange an MLP-in weight from the logical order [gate (F rows);
 * up (F rows)] into the packed order the library reads: blocks of 256 rows, block j =
 * [gate rows 128j .. 128j+127 ; up rows 128j .. 128j+127].  src_dev and dst_dev are
 * [2F, cols] bf16 device buffers that must not overlap; F % 128 == 0, F <= 2^19,
 * cols % 8 == 0, cols <= 2^20.  For a single-stream qkv_mlp
 * weight, pack its last 2F rows (pointer offset 3H * cols elements) and copy the first
 * 3H rows unchanged. */
dit_status dit_pack_mlp_in(const void* src_dev, void* dst_dev, int mlp_hidden, int cols, dit_stream_t stream);

/* Weight preparation for the e4m3 path: for each row r of w_dev [rows, cols] (bf16),
 * scale_dev[r] = max|w[r, :]| / 448 and q_dev[r, c] = e4m3(w[r, c] / scale[r]) (round to
 * nearest, saturating).  q_dev [rows, cols] bytes, scale_dev [rows] fp32; cols % 16 == 0,
 * rows and cols <= 2^20. */
dit_status dit_quantize_rows_fp8(const void* w_dev, int rows, int cols, void* q_dev, float* scale_dev,
                                 dit_stream_t stream);

/* Global modulation of one step ("flux2-klein-p100a" Caveats: computed once per step and
 * shared by all blocks).  tau = 1000 * sigma; s = [cos(tau f_k) | sin(tau f_k)],
 * f_k = 10000^(-k/128), k < 128; e = t_out SiLU(t_in s); m = mod SiLU(e).
 * sigma_dev [batch] fp32 device; mod_dev [batch, 17H] bf16 device, slots in order
 * img-dual (shift_a, scale_a, gate_a, shift_m, scale_m, gate_m), txt-dual (same six),
 * single (shift, scale, gate), final (shift, scale).  Uses the workspace as scratch. */
dit_status dit_modulation(const dit_weights* w, const float* sigma_dev, int batch, void* mod_dev, void* ws,
                          size_t ws_bytes, dit_stream_t stream);

/* One dual-stream block `layer` (0 <= layer < n_dual), in place on x_dev [B, N, H]
 * (rows text | image | reference).  Sources: "tt_flux2_klein -- Python reference",
 * Modules (tt_dit.py: the 5 dual-stream blocks, each with its own text and image weights)
 * and "Things that are easy to get wrong" (the joint sequence and RoPE); "flux2-klein-p100a"
 * Caveats (all 512 padded text rows, no mask; modulation global per step).  The block maths
 * is not written on the pages: the form below is the library's reading.  Per stream s
 * (text rows use `txt`, image and reference rows use `img` weights and modulation):
 *   y = (1 + scale_a) LN(x) + shift_a;  q, k, v = y qkv^T;  q, k <- RMSNorm_head * w;
 *   q, k <- RoPE;  o = joint softmax attention over all N rows, no mask;
 *   x += gate_a (o out^T);  y = (1 + scale_m) LN(x) + shift_m;
 *   x += gate_m (silu(y gate^T) * (y up^T)) mlp_out^T.
 * mod_dev [B, 17H] from dit_modulation; rope_dev [N, 64, 2] from dit_rope_table. */
dit_status dit_dual_block_fwd(const dit_weights* w, int layer, const dit_shape* shape, void* x_dev,
                              const void* mod_dev, const float* rope_dev, void* ws, size_t ws_bytes,
                              dit_stream_t stream);

/* One single-stream block `layer` (0 <= layer < n_single), in place on x_dev [B, N, H].
 * Sources: "tt_flux2_klein -- Python reference", Modules (tt_dit.py: the 20 single-stream
 * blocks, one weight set over the joint sequence) and "Things that are easy to get wrong";
 * "flux2-klein-p100a" Caveats (modulation global per step).  The fused projection's column
 * order is the library's reading:
 *   y = (1 + scale) LN(x) + shift;  [q | k | v | gate | up] = y qkv_mlp^T;
 *   q, k <- RMSNorm_head * w, RoPE;  o = attention;  act = silu(gate) * up;
 *   x += gate_s ([o | act] out^T).  Other arguments as dit_dual_block_fwd. */
dit_status dit_single_block_fwd(const dit_weights* w, int layer, const dit_shape* shape, void* x_dev,
                                const void* mod_dev, const float* rope_dev, void* ws, size_t ws_bytes,
                                dit_stream_t stream);

/* One whole DiT step (one velocity evaluation; "flux2-klein-p100a" task table: each of the
 * 4 steps is one DiT call, guidance 1.0, no CFG; "tt_flux2_klein -- Python reference",
 * Lower-level entry points: denoise consumes encode()'s [512, 7680] text features and the
 * reference tokens; Modules: tt_dit.py): modulation from sigma, embedders
 * (img/ref tokens by x_emb, text by ctx_emb) into the joint stream, n_dual dual blocks,
 * n_single single blocks, then the final layer (1 + scale_f) LN(x) + shift_f and
 * proj_out on the target-image rows only.
 * img_tokens [B, n_img, C], ref_tokens [B, n_ref, C] (NULL iff n_ref == 0),
 * txt_emb [B, n_txt, txt_dim], rope_dev [N, 64, 2] fp32, sigma_dev [B] fp32,
 * velocity_out [B, n_img, C]; all device. */
dit_status dit_step_fwd(const dit_weights* w, const dit_shape* shape, const void* img_tokens,
                        const void* ref_tokens, const void* txt_emb, const float* rope_dev, const float* sigma_dev,
                        void* velocity_out, void* ws, size_t ws_bytes, dit_stream_t stream);

/* The denoising loop on the device ("flux2-klein-p100a" task table: steps fixed at 4, each
 * one DiT call, guidance 1.0; "tt_flux2_klein -- Python reference", Lower-level entry
 * points: denoise).  x_tokens [B, n_img, C] bf16 (device) holds the initial latent tokens
 * and receives the final ones.  For k = 0 .. steps-1: v_k = the DiT step at sigma_k;
 * x <- x + (sigma_{k+1} - sigma_k) v_k (flow-matching Euler update).  sigmas_host: steps + 1
 * host floats in [0, 1000] (one schedule for every batch row; the 4-step klein schedule
 * ends at 0), 1 <= steps <= 8.  The modulation of all steps is computed first in one pass
 * over its weights; the latent is carried in fp32 in the workspace between steps and the
 * Euler update runs in the final projection's epilogue.  Reference tokens and text
 * features are the same at every step.  Workspace: dit_workspace_size bytes. */
dit_status dit_denoise_fwd(const dit_weights* w, const dit_shape* shape, void* x_tokens, const void* ref_tokens,
                           const void* txt_emb, const float* rope_dev, const float* sigmas_host, int steps, void* ws,
                           size_t ws_bytes, dit_stream_t stream);

/* dit_step_fwd with HOST inputs and output: copies img_tokens, ref_tokens, txt_emb and
 * sigma (host, same layouts; pinned memory gives asynchronous copies) into the
 * workspace, runs the step and copies the velocity back to velocity_host, all on
 * `stream`.  The result is valid once the stream has completed. */
dit_status dit_step_host(const dit_weights* w, const dit_shape* shape, const void* img_tokens_host,
                         const void* ref_tokens_host, const void* txt_emb_host, const float* rope_dev,
                         const float* sigma_host, void* velocity_host, void* ws, size_t ws_bytes,
                         dit_stream_t stream);

/* Synchronise `stream`, read and clear the workspace's device status word.  Returns
 * DIT_ERR_TIMEOUT if a kernel gave up on a wait since the last call, else DIT_OK
 * (or DIT_ERR_CUDA if the stream reports an error).  *where_out (may be NULL) receives
 * the id of the first wait that gave up. */
dit_status dit_sync_status(void* ws, dit_stream_t stream, uint32_t* where_out);

/* ---- CUDA graphs of a step (fixed shape and buffers) ------------------------------ */

/* A captured, instantiated CUDA graph of one dit_step_fwd (host_io == 0) or one
 * dit_step_host (host_io != 0) call with exactly these arguments: the same buffers are
 * read and written on every launch (their contents may change between launches; for
 * host_io the host buffers must be pinned).  Replaying it enqueues the whole step with one
 * call instead of ~125, which matters when the caller synchronises after every step (the
 * served path of the pages runs its compiled DiT inside CUDA-graph buckets for 1024², "FLUX.2
 * [klein] 4B/9B + Z-Image-Turbo on a shared DiT scaffold", Known gaps).  Creation runs the
 * step once on `stream` (warm-up), synchronises it, then captures; no other work may be
 * enqueued on `stream` meanwhile.  The handle owns the graph; the buffers stay
 * caller-owned and must outlive it.  Errors as for the step call, DIT_ERR_CUDA if capture
 * or instantiation fails. */
typedef struct dit_graph_s* dit_graph;
dit_status dit_step_graph_create(const dit_weights* w, const dit_shape* shape, const void* img_tokens,
                                 const void* ref_tokens, const void* txt_emb, const float* rope_dev,
                                 const float* sigma, void* velocity_out, void* ws, size_t ws_bytes, int host_io,
                                 dit_stream_t stream, dit_graph* graph_out);
/* Enqueue one replay of the graph on `stream`. */
dit_status dit_graph_launch(dit_graph graph, dit_stream_t stream);
/* Release the graph (NULL is accepted). */
dit_status dit_graph_destroy(dit_graph graph);

/* Failure-detection self-test: launches one kernel whose only thread waits on a device
 * barrier that nothing arrives on, with a limit of limit_us microseconds (1 .. 1e6).  The
 * bounded wait gives up, records DIT_ERR_TIMEOUT's bit and the site id 0x901 in the
 * workspace status word, and the kernel returns: dit_sync_status then reports
 * DIT_ERR_TIMEOUT and the context stays usable.  ws: any workspace of >= 256 bytes. */
dit_status dit_selftest_wait_timeout(void* ws, size_t ws_bytes, unsigned int limit_us, dit_stream_t stream);

/* ---- Component operations (the kernels a block is made of) ---------------------- */

/* Adaptive LayerNorm on rows of x: for batch b and row r < rows,
 * y[b, r] = (1 + scale_b) LN(x[b, x_row0 + r]) + shift_b, LN without affine, biased
 * variance, eps from the argument, statistics in fp32.  Rows r < split use
 * (shift_lo, scale_lo), the others (shift_hi, scale_hi); each vector [hidden] lives at
 * pointer + b * mod_stride elements.  x_dev [B, x_rows, hidden], y_dev [B, rows, hidden].
 * batch <= 64 and rows <= 2^20, else DIT_ERR_INVALID_ARG. */
dit_status dit_adaln(int batch, int rows, int hidden, const void* x_dev, int x_rows, int x_row0, int split,
                     const void* shift_lo, const void* scale_lo, const void* shift_hi, const void* scale_hi,
                     long long mod_stride, float eps, void* y_dev, dit_stream_t stream);

typedef enum {
  DIT_EPI_STORE = 0,          /* out = A W^T                                        */
  DIT_EPI_GATED_RESIDUAL = 1, /* out += gate_b * (A W^T), gate at gate + b*gate_stride */
  DIT_EPI_SWIGLU = 2          /* out = silu(A Wg^T) * (A Wu^T), W packed (2*n_out rows) */
} dit_epilogue;

/* Linear layer on the tensor cores: a_dev [B, rows, k], w_dev [n_w, k] (n_w = n_out,
 * or 2*n_out packed for SWIGLU), out_dev [B, rows, ld_out] written at columns
 * [0, n_out).  k % 8 == 0, n_out % 32 == 0 (SWIGLU: n_out % 128 == 0), ld_out % 8 == 0;
 * batch <= 64 and rows, n_out, k <= 2^20 (the token limit), else DIT_ERR_INVALID_ARG.
 * ws: any workspace of >= 256 bytes (only its status word is used). */
dit_status dit_linear(int batch, int rows, int n_out, int k, const void* a_dev, const void* w_dev, void* out_dev,
                      int ld_out, dit_epilogue epi, const void* gate_dev, long long gate_stride, void* ws,
                      size_t ws_bytes, dit_stream_t stream);

/* Joint attention: q/k/v_dev [B, heads, n, 128] bf16 (head-major), softmax over all n
 * keys with scale 1/sqrt(128), no mask; out_dev [B, n, ld_out] with head h written at
 * columns [128h, 128h + 128).  ld_out % 8 == 0, ld_out >= 128 * heads; batch <= 64,
 * n <= 2^20, heads <= 8192, else DIT_ERR_INVALID_ARG.  ws: any
 * workspace of >= 256 bytes (only its status word is used). */
dit_status dit_attention(int batch, int heads, int n, const void* q_dev, const void* k_dev, const void* v_dev,
                         void* out_dev, int ld_out, void* ws, size_t ws_bytes, dit_stream_t stream);

/* ---- Allocation-free variant -------------------------------------------------------- */

/* dit_modulation without a workspace, for callers that cannot allocate device memory
 * where they run the modulation: a plugin inside a host framework that owns every device
 * buffer and hands the plugin only its input and output tensors, or a serving loop that
 * forbids allocation after start-up (cudaMalloc can synchronise the device and can fail
 * once memory is fragmented).  The pages have no counterpart of this entry point; it
 * computes what dit_modulation computes.  Its fp32 scratch (two [batch, hidden] vectors)
 * lives in a fixed __device__ array of the library, 256 KB, which every GPU that loads the
 * library holds until the process exits; so batch <= 8 and hidden <= 4096, and larger
 * sizes return DIT_ERR_UNSUPPORTED with nothing launched.  The caller still passes
 * sigma_dev [batch] fp32 and mod_dev [batch, 17H] bf16 (device).  The first call on a
 * device looks up the array's device address (cudaGetSymbolAddress) with that device
 * current: make that first call before any stream capture.  Every call shares the one
 * array, so calls that overlap on the GPU (on different streams) race on it.  It never
 * calls cudaMalloc, cudaFree or an allocating library routine. */
dit_status dit_modulation_static(const dit_weights* w, const float* sigma_dev, int batch, void* mod_dev,
                                 dit_stream_t stream);

/* ---- Measurement ------------------------------------------------------------------ */

/* Kernel launches issued by this library since it was loaded (all entry points). */
unsigned long long dit_launch_count(void);

/* Start recording a CUDA event pair around every kernel launch (up to max_records
 * launches), tagged with the kernel's class (dit_kernel_class_name).  Events are
 * recorded on the launch's own stream.  A step captured by dit_step_graph_create while
 * recording is on carries its event pairs as event-record nodes: each replay records them
 * again (the records then hold the latest replay's times), so destroy such a graph before
 * the next dit_timing_begin, which releases the events. */
dit_status dit_timing_begin(int max_records);

/* Restrict the event pairs of dit_timing_begin to launches whose class bit is set in
 * class_mask (bit c = class c; ~0u, the initial value, records every class), so that a
 * timed region pays for events only around the kernels it measures.  Takes effect for
 * launches issued after the call.  Returns DIT_ERR_INVALID_ARG for a zero mask. */
dit_status dit_timing_select(unsigned int class_mask);

/* Stop recording, synchronise the recorded events and return up to `cap` records:
 * classes[i] and ms[i] (device time of launch i).  *n receives the count. */
dit_status dit_timing_end(int* n, int* classes, float* ms, int cap);

/* Static name of a kernel class id, or "?" for an unknown id. */
const char* dit_kernel_class_name(int cls);

#ifdef __cplusplus
}
#endif

#endif /* DIT_H_ */
