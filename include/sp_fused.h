/*
 * sp_fused.h — C boundary of the GB300 (sm_103a) library for the per-token stage of the
 * sequence-parallel rewrite
 *
 *     AllReduce -> RMSNorm -> quant   ==>   ReduceScatter -> RMSNorm -> quant -> AllGather
 *
 * On one GPU the tp partial-sum tensors that a ReduceScatter would reduce are plain device
 * buffers; the library sums them, adds bias and residual, applies RMSNorm with a weight, writes
 * the new residual and emits bf16, FP8-E4M3 (static per-tensor or per-token dynamic) or NVFP4
 * output, with padding rows zeroed. Output rows are in token order, which on one device is the
 * shard-contiguous layout an AllGather along the token dimension would produce.
 *
 * Sources (web pages; cited by title and section):
 *   "vllm-ascend SP / FlashComm1 / FlashComm2" (ai6s.net): §2.1 the AR -> RS + norm + AG rewrite;
 *       §2.2 its mathematical equivalence; §2.3 the add-RMSNorm-bias pattern and its replacement
 *       (reduce_scatter, chunk the residual, add + RMSNorm with weight and bias slot, all_gather);
 *       §2.4 token count padded to a multiple of tp; §3.3 pad -> reduce_scatter(dim 0) ... ->
 *       all_gather(dim 0) -> unpad.
 *   "vLLM SP / AsyncTP / quantization tech notes" (beaiera.top): §四 the static FP8 and NVFP4
 *       patterns (RS -> RMSNorm(local) -> quant(local) -> AG) and the per-tensor correctness
 *       table (static per-tensor, per-token and per-block scales are shard-local; dynamic
 *       per-tensor is not).
 *   "vllm-ascend PR #18671 解读: GLM V1 SP layout through DSA-CP": §2 contiguous token shards
 *       (3500 tokens padded to 3504, 219 per rank at TP=16); §5.2 shard checks that raise on a
 *       mismatch and zeroing of padding rows; §5.3 tail padding rows zeroed after the reduction.
 *   "基于Atlas A3集群的LongCat-Flash模型推理性能优化实践": o_proj TP paragraph (reduce_scatter =
 *       element-wise sum, then split along the batch/token dimension).
 *
 * Conventions for every entry point:
 *   - All tensor arguments are DEVICE pointers into the memory of the current CUDA device, unless
 *     the argument says "host". The caller owns every buffer; the library allocates nothing and
 *     may be called concurrently from several host threads. What it keeps between calls is
 *     listed where it is used: the device error word (sp_device_error), the dynamic row
 *     schedule's per-stream counters with their completion numbers and the one stream it creates
 *     to read those back (sp_fused_options.schedule), the no-allocation entry's counter
 *     (sp_fused_reduce_norm_noalloc) and each host thread's last launch (sp_last_launch).
 *   - bf16 is IEEE binary32's top 16 bits; FP8 E4M3 is the OCP "E4M3" (fn) format; E2M1 is the
 *     OCP MX FP4 format. All tensors are dense, row-major, C-contiguous.
 *   - Calls are asynchronous on `stream` (NULL = legacy default stream); nothing synchronises the
 *     host, except that a dynamic-schedule call on a new stream that finds all 256 counter slots
 *     taken waits for a 2 KB read on the library's own stream (sp_fused_options.schedule).
 *     Errors found before the launch leave every buffer untouched.
 */
#ifndef SP_FUSED_H
#define SP_FUSED_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t, so CUDA callers pass their stream directly. */
typedef struct CUstream_st* sp_stream_t;

typedef enum sp_status {
  SP_OK = 0,
  SP_ERR_INVALID_ARG = 1,  /* a shape, mode, eps, pointer or overlap rule is broken */
  SP_ERR_UNSUPPORTED = 2,  /* well-formed but not provided (dynamic per-tensor FP8; H too large) */
  SP_ERR_ALIGNMENT = 3,    /* a device pointer is not 16-byte aligned */
  SP_ERR_CUDA = 4          /* the CUDA runtime reported an error (launch or attribute query) */
} sp_status;

typedef enum sp_quant_mode {
  SP_QUANT_NONE = 0,             /* out: bf16 [T_pad][H] */
  SP_QUANT_FP8_STATIC = 1,       /* out: e4m3 [T_pad][H]; q = E4M3(y / scale[0]) */
  SP_QUANT_FP8_PER_TOKEN = 2,    /* out: e4m3 [T_pad][H]; out_scales: fp32 [T_pad], s_t = max|y_t|/448 */
  SP_QUANT_NVFP4 = 3,            /* out: e2m1 packed [T_pad][H/2]; out_scales: e4m3 [T_pad][H/16] */
  SP_QUANT_FP8_DYNAMIC_PER_TENSOR = 4 /* always SP_ERR_UNSUPPORTED: its scale is not shard-local */
} sp_quant_mode;

/*
 * sp_fused_reduce_norm — the whole per-token stage in one pass over HBM.
 *
 * For every row t < T_valid (h, y are fp32 vectors of length H):
 *   h            = sum_{r<tp} partials[r][t] + bias + residual[t]     (the ReduceScatter sum)
 *   residual_out[t] = bf16_rn(h)                                      (the new residual)
 *   y            = h * rsqrt(mean(h^2) + eps) * weight                  (RMSNorm, per token)
 *   out[t]       = by quant_mode:
 *     NONE           bf16_rn(y)
 *     FP8_STATIC     e4m3_satfinite_rn(y / scale[0])        (scale = dequantisation scale)
 *     FP8_PER_TOKEN  s_t = max_j|y_j| / 448 -> out_scales[t] (fp32);
 *                    e4m3_satfinite_rn(y / s_t), all zero when s_t == 0
 *     NVFP4          per 16-element block b of the row: sf_b = e4m3_satfinite_rn(gs * max|y_b| / 6)
 *                    -> out_scales[t][b]; q = e2m1_satfinite_rn(y * gs / sf_b), zero when
 *                    sf_b == 0; gs = scale[0] (an encode multiplier); element 2i of the row goes
 *                    to the low nibble of byte i, 2i+1 to the high nibble.
 * Rows t >= T_valid are padding: none of their inputs is read and every byte of their out,
 * out_scales and residual_out rows is written as zero.
 *
 * Restates: the sum over partials is the ReduceScatter's element-wise sum split along tokens
 * (LongCat-Flash A3 page, o_proj TP paragraph; vllm-ascend SP/FlashComm notes §2.1-§2.2); bias,
 * residual, new residual and RMSNorm with weight follow the add-RMSNorm-bias replacement
 * (vllm-ascend SP/FlashComm notes §2.3); the quantisers are the local quant after the norm and
 * their shard-local scales (vLLM SP/AsyncTP/quant notes §四); T_pad is the token count padded to
 * a multiple of tp (vllm-ascend SP/FlashComm notes §2.4) and padding rows are zeroed after the
 * reduction (PR #18671 notes §5.2-§5.3).
 *
 * Arguments:
 *   partials     bf16 [tp][T_pad][H]: partial r holds rank r's un-reduced output for every token.
 *   tp           number of partials, >= 1.
 *   T_pad        padded token count, a multiple of tp (shard r = rows [r*T_pad/tp, (r+1)*T_pad/tp)).
 *   T_valid      real tokens, 0 <= T_valid <= T_pad.
 *   H            hidden size, > 0, multiple of 8 (of 16 for NVFP4), at most sp_max_hidden().
 *   residual     bf16 [T_pad][H], or NULL for a first layer with no incoming residual.
 *   weight       bf16 [H] RMSNorm weight.
 *   bias         bf16 [H] added once after the reduction, or NULL.
 *   eps          > 0 and finite.
 *   quant_mode   an sp_quant_mode.
 *   scale        device pointer to one fp32: the static FP8 scale (> 0) or the NVFP4 global
 *                scale gs (> 0); may be NULL for NONE and FP8_PER_TOKEN. Its value is read on
 *                the device and is not checked.
 *   out          see quant_mode.
 *   out_scales   NULL for NONE and FP8_STATIC; fp32 [T_pad] for FP8_PER_TOKEN; e4m3
 *                [T_pad][H/16] (row-major, one byte per block) for NVFP4.
 *   residual_out bf16 [T_pad][H]; may be exactly `residual` (updated in place), otherwise it
 *                must not overlap any input.
 *   stream       CUDA stream of the launch.
 * Every non-NULL pointer must be 16-byte aligned (SP_ERR_ALIGNMENT). No output may overlap an
 * input or another output (SP_ERR_INVALID_ARG), except residual_out == residual.
 * Checks run in this order and the first failure is returned: quant_mode, shapes (tp, T_pad,
 * T_valid, H, and tp * T_pad * H * 2 <= 2^62 bytes), eps, required pointers, overlaps,
 * alignment, H <= sp_max_hidden(). T_pad == 0 is a valid call that launches nothing.
 * Returns SP_OK once the kernel is enqueued, or the failed check's status, or SP_ERR_CUDA.
 */
sp_status sp_fused_reduce_norm(const void* partials, int tp, int64_t T_pad, int64_t T_valid,
                               int64_t H, const void* residual, const void* weight,
                               const void* bias, float eps, int quant_mode, const float* scale,
                               void* out, void* out_scales, void* residual_out,
                               sp_stream_t stream);

/*
 * sp_check_args — the argument checks of sp_fused_reduce_norm alone, in the same order and with
 * the same statuses. Pointers are only compared, never dereferenced; touches no GPU and needs
 * no CUDA device. The shape rules are the single-GPU form of the shard checks that raise on a
 * layout mismatch (PR #18671 notes §5.2); the refusal of dynamic per-tensor FP8 is the
 * per-tensor correctness table (vLLM SP/AsyncTP/quant notes §四).
 */
sp_status sp_check_args(const void* partials, int tp, int64_t T_pad, int64_t T_valid, int64_t H,
                        const void* residual, const void* weight, const void* bias, float eps,
                        int quant_mode, const float* scale, const void* out,
                        const void* out_scales, const void* residual_out);

/*
 * Options of sp_fused_reduce_norm_ex. Initialise with sp_options_init (which gives exactly
 * sp_fused_reduce_norm) and change what is needed.
 *   partial_scale  every partial is multiplied by this before the reduction (a per-rank output
 *                  scale applied before the ReduceScatter, PR #18671 notes §5.3): finite; 1 = none.
 *   addend         bf16 [T_pad][H] added after the reduction and before the norm, and so also
 *                  part of the new residual: h = partial_scale * sum_r partials[r][t] + bias +
 *                  residual[t] + addend[t] (the per-shard extra input of the Qwen3-VL deepstack
 *                  rewrite, vllm-ascend SP notes §2.3); NULL = none. Never read on padding rows.
 *   scale_layout   NVFP4 block scales: SP_SCALES_ROW_MAJOR ([T_pad][H/16], one byte per block)
 *                  or SP_SCALES_SWIZZLED_128X4, the layout block-scaled GEMMs read: the
 *                  [T_pad][H/16] scale matrix padded to R = ceil(T_pad/128)*128 rows and
 *                  C = ceil(H/64)*4 columns (padding bytes written as zero), stored as 512-byte
 *                  tiles of 128 rows x 4 columns, tile (i, j) at byte (i * C/4 + j) * 512 and row r,
 *                  column c of a tile at (r % 32) * 16 + (r / 32) * 4 + c; out_scales then holds
 *                  R * C bytes (sp_out_scales_bytes_ex). SWIZZLED with another mode is
 *                  SP_ERR_INVALID_ARG; any other value SP_ERR_UNSUPPORTED.
 *   host_buffers   0: every tensor is in device memory; 1: tensors are in page-locked host memory
 *                  (or device memory) and are read/written across the host link (zero-copy).
 *   schedule       how rows reach CTAs; the results are the same bytes either way.
 *                  SP_SCHEDULE_STATIC: CTA b takes rows b, b + grid, b + 2*grid, ...
 *                  SP_SCHEDULE_DYNAMIC: CTA b takes row b, then claims further rows from a row
 *                  counter of the call's stream, so CTAs that get more memory bandwidth take more
 *                  rows (applies to the staged kernel, the one device-buffer calls use).
 *                  SP_SCHEDULE_AUTO (the default): dynamic when the staged kernel gives every CTA
 *                  at least 10 rows, H >= 2048 and (tp + 3) * 2H >= 24 KB, static otherwise.
 *                  Without row_counter (below) the counters are a fixed table of 256 slots in
 *                  the library's device memory (no allocation): one slot per stream (told apart
 *                  by cudaStreamGetId), reset by each call's last CTA, so calls on one stream
 *                  reuse it in stream order and calls on different streams never share one.
 *                  Once all 256 are taken, a call on a new stream takes over the least
 *                  recently used idle slot: one whose launches have all finished with it (each
 *                  launch records that in the library's device memory; the library reads the
 *                  table back on a non-blocking stream of its own, created the first time, only
 *                  when a new stream finds the table full). Only while every slot still has a
 *                  launch queued or claiming rows does a call on a new stream run the static
 *                  schedule (same results, up to ~13 % slower on large calls), unless it passes
 *                  row_counter. A call also falls back to the static schedule while its stream
 *                  is being captured into a CUDA graph (a replay may run beside calls on the
 *                  capturing stream), again unless it passes row_counter. sp_last_launch tells
 *                  which schedule a call ran. Any other value is SP_ERR_UNSUPPORTED.
 *   launch         a launch configuration (below) to run instead of the one sp_select_launch
 *                  picks, for tests and tuning; NULL (the default) = the library's choice. The
 *                  checks of sp_fused_reduce_norm_with_config apply. With host_buffers = 1 it
 *                  must name the DIRECT kernel (else SP_ERR_UNSUPPORTED).
 *   row_counter    NULL (the default), or the caller's own device buffer of two uint32 (8 bytes,
 *                  16-byte aligned, zero before its first use) that the dynamic schedule claims
 *                  rows from instead of the library's per-stream table. Each call leaves it zero
 *                  when it completes, so it can be reused by calls that are ordered one after the
 *                  other (one stream, or graph replays that do not overlap); calls that overlap
 *                  on the GPU must not share one. Used also while the stream is being captured.
 *                  After a call whose status reports a timeout, zero it again before reuse.
 *   status         NULL (the default), or a device uint32 (16-byte aligned) that the call ORs
 *                  its device-side error bits into (SP_DEVICE_ERR_WAIT_TIMEOUT) in place of the
 *                  device error word of sp_device_error, in stream order: read it once the
 *                  call's work on the stream has completed (a copy on the same stream, or after
 *                  a synchronisation). The library never clears it. When a bit is set, that
 *                  call's outputs are undefined.
 *                  row_counter and status may not overlap any input or output of the call.
 */
enum { SP_SCALES_ROW_MAJOR = 0, SP_SCALES_SWIZZLED_128X4 = 1 };
enum { SP_SCHEDULE_AUTO = 0, SP_SCHEDULE_STATIC = 1, SP_SCHEDULE_DYNAMIC = 2 };

struct sp_launch_config;

typedef struct sp_fused_options {
  float partial_scale;
  const void* addend;
  int scale_layout;
  int host_buffers;
  int schedule;
  const struct sp_launch_config* launch;
  void* row_counter;
  uint32_t* status;
} sp_fused_options;

/* sp_options_init — the defaults (exactly sp_fused_reduce_norm). The options restate PR #18671
 * notes §5.3 (partial_scale) and vllm-ascend SP/FlashComm notes §2.3 (addend). */
void sp_options_init(sp_fused_options* options /* host, out */);

/*
 * sp_fused_reduce_norm_ex — sp_fused_reduce_norm with options (NULL options = defaults). The
 * addend follows the same rules as the residual (16-byte aligned, may not overlap an output).
 * A non-finite partial_scale is SP_ERR_INVALID_ARG. Restates, beyond sp_fused_reduce_norm: the
 * output scale applied to each rank's partial before the ReduceScatter (PR #18671 notes §5.3) and
 * the per-shard addend added after it (vllm-ascend SP/FlashComm notes §2.3, deepstack rewrite).
 */
sp_status sp_fused_reduce_norm_ex(const sp_fused_options* options /* host */,
                                  const void* partials, int tp, int64_t T_pad, int64_t T_valid,
                                  int64_t H, const void* residual, const void* weight,
                                  const void* bias, float eps, int quant_mode, const float* scale,
                                  void* out, void* out_scales, void* residual_out,
                                  sp_stream_t stream);

/* sp_check_args_ex — the checks of sp_fused_reduce_norm_ex alone (no GPU needed); the same
 * passages as sp_check_args (PR #18671 notes §5.2) plus the option rules above. */
sp_status sp_check_args_ex(const sp_fused_options* options /* host */, const void* partials,
                           int tp, int64_t T_pad, int64_t T_valid, int64_t H, const void* residual,
                           const void* weight, const void* bias, float eps, int quant_mode,
                           const float* scale, const void* out, const void* out_scales,
                           const void* residual_out);

/*
 * sp_fused_reduce_norm_host — the same stage, with every tensor argument (partials, residual,
 * weight, bias, scale, out, out_scales, residual_out) in page-locked HOST memory (cudaHostAlloc
 * or cudaHostRegister; device memory is accepted too). The kernel reads the inputs across the
 * host link and writes the outputs back across it as it goes (zero-copy), so the host->device
 * and device->host traffic of a call overlap each other and the computation, with no device
 * staging buffers. Same arguments, checks, statuses and results as sp_fused_reduce_norm, plus
 * SP_ERR_INVALID_ARG for a pointer the device cannot reach (pageable memory). Asynchronous on
 * `stream`: synchronise the stream before reading the outputs on the host. The stage is the one
 * sp_fused_reduce_norm restates (vllm-ascend SP/FlashComm notes §2.3; vLLM SP/AsyncTP/quant
 * notes §四); host-resident buffers have no counterpart on the pages.
 */
sp_status sp_fused_reduce_norm_host(const void* partials, int tp, int64_t T_pad, int64_t T_valid,
                                    int64_t H, const void* residual, const void* weight,
                                    const void* bias, float eps, int quant_mode,
                                    const float* scale, void* out, void* out_scales,
                                    void* residual_out, sp_stream_t stream);

/*
 * sp_fused_reduce_norm_noalloc — sp_fused_reduce_norm for callers that may not allocate device
 * memory. Some code cannot call cudaMalloc or any allocating routine at the point where it runs
 * this stage: code recording a CUDA graph (allocation is not a capturable operation), a plugin
 * or custom operator whose host framework owns every device buffer and hands out only the
 * tensors of the call, and latency-critical serving loops that forbid allocation after start-up
 * (cudaMalloc can synchronise the device and take milliseconds). Such a caller cannot provide
 * the 8-byte row counter that the dynamic row schedule needs (sp_fused_options.row_counter), and
 * the library's per-stream counter table serves no call under graph capture and at most 256
 * streams with launches in flight at once. This
 * entry point keeps that counter in an array of the library's own static device memory instead:
 * 8 bytes, one array per GPU that loads the library, held until the process exits, shared by
 * every call of this entry point. The caller passes exactly the buffers of sp_fused_reduce_norm.
 *
 * Same arguments, checks, statuses, launch choice and results (byte for byte) as
 * sp_fused_reduce_norm; nothing is allocated, by the library or on its behalf. Before its launch
 * it clears the counter on `stream` (cudaMemsetAsync of the 8 bytes), since the array keeps what
 * the previous call left. The first call on a device looks up the array's device address with
 * cudaGetSymbolAddress; make that first call before any stream capture on that device. Calls of
 * this entry point that overlap on the GPU (on different streams, or in graph replays that run at
 * the same time) share the one counter and race: order them, for instance on one stream.
 * Maximum: T_pad up to 2^31 - 2^16 rows, the range of the 32-bit counter; larger calls return
 * SP_ERR_UNSUPPORTED before anything is enqueued. The pages have no counterpart of this entry
 * point (it concerns memory management only): no counterpart on the pages.
 */
sp_status sp_fused_reduce_norm_noalloc(const void* partials, int tp, int64_t T_pad,
                                       int64_t T_valid, int64_t H, const void* residual,
                                       const void* weight, const void* bias, float eps,
                                       int quant_mode, const float* scale, void* out,
                                       void* out_scales, void* residual_out, sp_stream_t stream);

/*
 * Launch configurations. sp_fused_reduce_norm picks one by itself (sp_select_launch tells
 * which); sp_fused_reduce_norm_with_config runs a given one, for tests and tuning. Every
 * configuration computes the same function.
 *   kernel        SP_KERNEL_STAGED: one CTA per row at a time; a producer thread streams the
 *                 row's tp partial rows and residual row from HBM into a shared-memory ring with
 *                 bulk asynchronous copies (cp.async.bulk + mbarrier), consumer warps reduce
 *                 from shared memory. With split > 1 (one vector per thread): one cluster of
 *                 `split` CTAs per row, every row at once (grid = split x T rows), each CTA
 *                 bringing its slice of all the row's segments into shared memory with one bulk
 *                 copy each (no ring; stages and ctas_per_sm are ignored); a slice of every
 *                 segment must fit one CTA's shared memory (else SP_ERR_UNSUPPORTED).
 *                 SP_KERNEL_DIRECT: the same CTA-per-row mapping with 128-bit loads straight into
 *                 registers.
 *   vec_per_thread  16-byte vectors (8 elements) of a row that each consumer thread owns: 1, 2, 4.
 *   ctas_per_sm     CTAs per SM the grid is sized for: grid = SMs x min(ctas_per_sm, CTAs of
 *                   this kernel an SM can hold), capped at T_pad; 1 .. 32.
 *   stages          shared-memory ring depth in row segments of 2*H bytes (STAGED only); 0 picks
 *                   the deepest ring that fits ctas_per_sm CTAs on an SM.
 *   split           CTAs that share each row: 0 or 1, a row per CTA; 2, 4 or 8, a thread-block
 *                   cluster of that many CTAs per row, each owning a contiguous slice of it and
 *                   combining the row's sum of squares (and max) through distributed shared
 *                   memory, so that a call with few rows uses `split` times as many SMs. DIRECT
 *                   (vec_per_thread 1 or 2): grid = split x min(T rows, SMs x ctas_per_sm /
 *                   split) CTAs; STAGED (vec_per_thread 1): see above. Another value is
 *                   SP_ERR_INVALID_ARG; split > 1 with vec_per_thread 4, or with the STAGED kernel
 *                   at vec_per_thread 2, is SP_ERR_UNSUPPORTED.
 * Launch shapes are this library's choice for GB300 and have no counterpart on the pages (their
 * fused operators are Ascend kernels); the function computed is sp_fused_reduce_norm's.
 */
enum { SP_KERNEL_STAGED = 0, SP_KERNEL_DIRECT = 1 };

typedef struct sp_launch_config {
  int kernel;
  int vec_per_thread;
  int ctas_per_sm;
  int stages;
  int split;
} sp_launch_config;

sp_status sp_select_launch(int tp, int64_t T_pad, int64_t H, int quant_mode,
                           sp_launch_config* config /* host, out */);

sp_status sp_fused_reduce_norm_with_config(const sp_launch_config* config /* host */,
                                           const void* partials, int tp, int64_t T_pad,
                                           int64_t T_valid, int64_t H, const void* residual,
                                           const void* weight, const void* bias, float eps,
                                           int quant_mode, const float* scale, void* out,
                                           void* out_scales, void* residual_out,
                                           sp_stream_t stream);

/*
 * sp_last_launch — what the calling thread's last successful fused-stage call launched: the
 * configuration (stages resolved), the CTAs launched and the row schedule it ran
 * (SP_SCHEDULE_STATIC or SP_SCHEDULE_DYNAMIC; the direct kernel is always static). All zero
 * before the first such call on this thread. Host only; SP_ERR_INVALID_ARG for a NULL pointer.
 * Lets a caller see, for instance, that a call fell back to the static schedule. A utility with
 * no counterpart on the pages.
 */
typedef struct sp_launch_info {
  sp_launch_config config;
  int grid;
  int schedule;
} sp_launch_info;

sp_status sp_last_launch(sp_launch_info* info /* host, out */);

/*
 * Layout helpers (host only, no device use).
 *   sp_pad_tokens: the smallest multiple of tp that is >= T (token padding before the
 *       ReduceScatter; vllm-ascend SP notes §2.4, §3.3), or -1 if T < 0 or tp < 1.
 *   sp_shard_rows: rows [*start, *start + *len) of shard `rank` — the contiguous segment of
 *       T_pad/tp rows that rank owns (PR #18671 notes §2, §5.2); SP_ERR_INVALID_ARG when
 *       T_pad % tp != 0 or rank is out of range.
 *   sp_out_bytes / sp_out_scales_bytes(_ex): sizes of `out` and `out_scales` for a mode (and a
 *       scale layout; 0 for no buffer), or -1 for an invalid mode or layout.
 *   sp_max_hidden: the largest H the kernels take.
 * Buffer sizes follow the layouts of sp_fused_reduce_norm (vLLM SP/AsyncTP/quant notes §四 for
 * the per-token and per-block scales).
 */
int64_t sp_pad_tokens(int64_t T, int tp);
sp_status sp_shard_rows(int64_t T_pad, int tp, int rank, int64_t* start /* host */,
                        int64_t* len /* host */);
int64_t sp_out_bytes(int64_t T_pad, int64_t H, int quant_mode);
int64_t sp_out_scales_bytes(int64_t T_pad, int64_t H, int quant_mode);
int64_t sp_out_scales_bytes_ex(int64_t T_pad, int64_t H, int quant_mode, int scale_layout);
int64_t sp_max_hidden(void);

/*
 * FlashComm2 token reorganisation (vllm-ascend SP/FlashComm notes §4.2-4.4, worked example in
 * §4.4), all ranks on one GPU. With G = global_tp, P = otp_size, D = odp_size = G/P,
 * F = H/G, S = N/G:
 *   x  [G][N][F] elements of elem_bytes bytes: rank r's feature slice of all N tokens.
 *   y  [G][N/D][D*F]: what rank r = g*D + j holds after (1) every rank cuts its slice into D
 *      packets by the reorganised batch ids (packet j = token segments j, j+D, j+2D, ... of S
 *      tokens each), (2) the all_to_all inside ODP group {g*D .. g*D+D-1}, (3) the concat of the
 *      D received pieces along the feature dimension: y[r][k*S + t][m*F + f] =
 *      x[g*D + m][(j + k*D)*S + t][f]. The ranks {j, j+D, ...} (an OTP group) then hold the same
 *      tokens with complementary features.
 * Requirements: G, P >= 1, G % P == 0, N % G == 0, H % G == 0, elem_bytes in {1, 2, 4, 8},
 * N * H * elem_bytes <= 2^62 (SP_ERR_INVALID_ARG); x and y 16-byte aligned and F * elem_bytes a multiple of 16
 * (SP_ERR_ALIGNMENT); x and y must not overlap. N == 0 launches nothing. Device pointers,
 * asynchronous on `stream`.
 */
sp_status sp_fc2_reorganize(const void* x, int global_tp, int otp_size, int64_t N, int64_t H,
                            int elem_bytes, void* y, sp_stream_t stream);
sp_status sp_fc2_check_args(const void* x, int global_tp, int otp_size, int64_t N, int64_t H,
                            int elem_bytes, const void* y);
/* The reorganised batch ids: ids[j*P + k] = j + k*D (D lists of P segments; host array), the
 * reorgnized_batch_ids of vllm-ascend SP/FlashComm notes §4.4. */
sp_status sp_fc2_batch_ids(int global_tp, int otp_size, int* ids /* host, [D*P] */);

/* Name of a status code, e.g. "SP_ERR_ALIGNMENT"; "SP_UNKNOWN_STATUS" for other values. A
 * utility with no counterpart on the pages. */
const char* sp_status_string(int status);

/*
 * Device-side error word. The waits of the staged kernel and of the reorganisation kernel on
 * their shared-memory rings are bounded in time; a wait that runs out (which only a hardware or
 * runtime fault could cause) sets SP_DEVICE_ERR_WAIT_TIMEOUT here (or, for a call that passed a
 * status word in its options, in that word instead), abandons the launch after letting its
 * copies in flight land, and the rows (or output tiles) it had not finished hold undefined
 * values. sp_device_error reads (and, when `clear` is non-zero, resets) the word of
 * the current device; it synchronises with the device. SP_ERR_CUDA if the runtime call fails.
 * Failure reporting of this library, with no counterpart on the pages.
 */
enum { SP_DEVICE_ERR_WAIT_TIMEOUT = 1 };
sp_status sp_device_error(uint32_t* flags /* host, out */, int clear);

/*
 * sp_selftest_wait_timeout — exercises that timeout path on the current device: one warp waits,
 * with a limit of `limit_ns` (1 ns .. 2 s), on a shared-memory barrier that nothing completes;
 * the wait gives up, sets SP_DEVICE_ERR_WAIT_TIMEOUT in the device error word and the kernel
 * ends normally (the context stays usable). Asynchronous on `stream`; SP_ERR_INVALID_ARG for a
 * limit out of range. A test hook with no counterpart on the pages.
 */
sp_status sp_selftest_wait_timeout(uint64_t limit_ns, sp_stream_t stream);

/*
 * sp_selftest_fused_timeout — the fused stage's own abort path on the GPU, without a fault. The
 * call runs like sp_fused_reduce_norm_ex with `options` on the staged kernel with two vectors
 * per consumer thread (so H <= 8192; options->launch, if given, must name that kernel and
 * vec_per_thread 2; host_buffers must be 0; else SP_ERR_UNSUPPORTED), except that every bounded
 * wait of the launch
 * gives up after `limit_ns` (1 ns .. 2 s) and the producer of CTA 0 never fills ring stage number
 * `withhold` (counted from 0 in the order it fills stages: with the dynamic schedule each row's
 * first stage also carries its index) and issues nothing after it. The consumer warps' waits on
 * that stage run out, all of them leave together, the producer's drain of it runs out too, and
 * the launch ends with SP_DEVICE_ERR_WAIT_TIMEOUT in the options' status word (or, without one,
 * in the device error word); the context stays usable and the outputs are undefined. If CTA 0 fills fewer
 * stages than `withhold`, nothing runs out. Asynchronous on `stream`; SP_ERR_INVALID_ARG for a
 * limit out of range or a negative `withhold`. A test hook with no counterpart on the pages.
 */
sp_status sp_selftest_fused_timeout(uint64_t limit_ns, int64_t withhold,
                                    const sp_fused_options* options /* host */,
                                    const void* partials, int tp, int64_t T_pad, int64_t T_valid,
                                    int64_t H, const void* residual, const void* weight,
                                    const void* bias, float eps, int quant_mode,
                                    const float* scale, void* out, void* out_scales,
                                    void* residual_out, sp_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* SP_FUSED_H */
