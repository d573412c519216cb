/*
 * psv.h — C ABI of libpsv: single-GPU serving of autoregressive-denoising
 * DiT world models on GB300 (sm_103a).
 *
 * The problem these calls serve (AREX article "vLLM 与 Physis-AI 联合介绍
 * PhysisServe 推理系统", §难题 and §三层设计; BAAI announcement
 * "智源悟界·PhysisServe：首个兼顾智能与高频吞吐的物理 AI 推理系统",
 * §新一代物理 AI 的基础设施 Fig. 1 and §PhysisServe Fig. 2–3):
 *   - a stream produces latent chunks; every chunk starts from pure noise
 *     and is denoised over S steps;
 *   - at step s and transformer block b a chunk attends to its own tokens
 *     plus the still-noisy keys/values that the W preceding chunks left at
 *     the same (block, step), so chunk c step s may run once chunk c step
 *     s-1 and chunk c-1 step s are done;
 *   - every ready (chunk, step) task of every stream is time-shared on the
 *     one GPU: a "wave" runs them all, block by block, each block as one
 *     batched launch per operation (same-block batching, Fig. 3 right).
 *
 * Conventions
 *   - every call returns 0 (PSV_OK) or a negative PSV_E* code; on error
 *     psv_last_error() describes it; PSV_ECUDA and PSV_EDEVICE are sticky;
 *   - the library never frees caller memory; host inputs are copied before
 *     a call returns, so the caller may reuse its buffers at once;
 *   - device work is issued on the caller's CUDA stream (given at create)
 *     and is asynchronous unless a call says otherwise;
 *   - all matrices are row-major; linear weights use the [out, in] layout.
 */
#ifndef PSV_H
#define PSV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ------------------------------------------------------ */
#define PSV_OK          0
#define PSV_EINVAL     (-1)  /* bad argument, shape or state                   */
#define PSV_ENOMEM     (-2)  /* arena too small / host allocation failed       */
#define PSV_EAGAIN     (-3)  /* nothing to return yet / queue full: retry later */
#define PSV_ETIMEDOUT  (-4)  /* psv_sync deadline passed (host-side polling)    */
#define PSV_ECUDA      (-5)  /* a CUDA runtime call failed (sticky)             */
#define PSV_EDEVICE    (-6)  /* a kernel raised its error word (sticky)         */

/* ---- create flags -------------------------------------------------------- */
#define PSV_FLAG_PLAN_ONLY   1  /* host scheduler only: no device, no arena     */
#define PSV_FLAG_SEQUENTIAL  2  /* one task per wave, lowest (stream, chunk,
                                   step) first: strictly sequential order       */
#define PSV_FLAG_CHUNK_COND  4  /* reserve per-chunk conditioning tables, for
                                   psv_submit_chunk_cond                       */
#define PSV_FLAG_LATENCY     8  /* latency mode: a wave runs only each stream's
                                   oldest ready chunk, so a chunk goes through
                                   its S steps in S consecutive waves (response
                                   time S single-chunk waves instead of S full
                                   waves), at the cost of smaller batches      */

/* ---- model description --------------------------------------------------
 * B blocks, S Euler steps (t_s = 1 - s/S), model width d = H*dh, MLP width
 * F, latent channels C (already patchified), T tokens per chunk, KV window
 * W (a chunk sees its own KV plus that of the W preceding chunks).
 * Requirements: d % 128 == 0, F % 64 == 0, dh in {32, 64, 128}, T >= 1,
 * W >= 0, 1 <= S <= 8, t_embed % 2 == 0 and <= 1024, C <= 256.
 * max_inflight: chunks of one stream alive at once (submitted and not yet
 * polled); 0 selects S + 4. */
typedef struct psv_model_desc {
  int32_t B, S, d, H, dh, F, C, T, W;
  int32_t max_streams;
  int32_t max_inflight;
  int32_t t_embed;      /* sinusoidal timestep-embedding width (256)       */
  float   ln_eps;       /* LayerNorm epsilon (1e-6)                        */
  float   rope_theta;   /* RoPE base (1e4)                                 */
  int32_t flags;        /* PSV_FLAG_*                                      */
} psv_model_desc;

/* ---- weights --------------------------------------------------------------
 * Global tensors (block = -1):
 *   IN_W [d, C]  IN_B [d]        latent -> residual stream
 *   T1_W [d, t_embed] T1_B [d]   time MLP, first layer (SiLU after it)
 *   T2_W [d, d]  T2_B [d]        time MLP, second layer
 *   FMOD_W [2d, d] FMOD_B [2d]   final adaLN: [shift_f, scale_f]
 *   OUT_W [C, d] OUT_B [C]       velocity head
 * Per block b (block = b):
 *   QKV_W [3d, d] QKV_B [3d]     rows [q | k | v], head h = rows h*dh..
 *   O_W [d, d]   O_B [d]
 *   UP_W [F, d]  UP_B [F]        GELU (tanh form) after it
 *   DOWN_W [d, F] DOWN_B [d]
 *   MOD_W [6d, d] MOD_B [6d]     adaLN: [shift1, scale1, gate1, shift2,
 *                                scale2, gate2] = MOD_W SiLU(e_s) + MOD_B
 * Matrices are stored in bf16 (f32 input is rounded to nearest even);
 * biases are stored in f32.  All tensors must be loaded before
 * psv_open_stream. */
enum {
  PSV_W_IN_W = 0, PSV_W_IN_B, PSV_W_T1_W, PSV_W_T1_B, PSV_W_T2_W, PSV_W_T2_B,
  PSV_W_FMOD_W, PSV_W_FMOD_B, PSV_W_OUT_W, PSV_W_OUT_B,
  PSV_W_QKV_W = 16, PSV_W_QKV_B, PSV_W_O_W, PSV_W_O_B, PSV_W_UP_W, PSV_W_UP_B,
  PSV_W_DOWN_W, PSV_W_DOWN_B, PSV_W_MOD_W, PSV_W_MOD_B
};
#define PSV_DTYPE_F32   0
#define PSV_DTYPE_BF16  1
#define PSV_LOC_HOST    0
#define PSV_LOC_DEVICE  1

typedef struct psv_weight {
  int32_t id;          /* PSV_W_*                                   */
  int32_t block;       /* -1 for global tensors, else 0..B-1        */
  const void* data;    /* host or device pointer, see location      */
  int32_t dtype;       /* PSV_DTYPE_F32 or PSV_DTYPE_BF16           */
  int32_t location;    /* PSV_LOC_HOST or PSV_LOC_DEVICE            */
  int64_t numel;       /* must equal the tensor's element count     */
} psv_weight;

/* One scheduled task, for introspection (psv_wave_plan). */
typedef struct psv_task {
  int32_t stream;      /* stream id                                          */
  int32_t chunk;       /* chunk index c within the stream                    */
  int32_t step;        /* denoising step s                                   */
  int32_t slot;        /* KV ring slot the task writes: c mod (W+1)          */
  int32_t kv_len;      /* keys the task attends to: (min(c, W) + 1) * T      */
  int32_t row_off;     /* first row of the task in the wave's batch          */
  int32_t state_slot;  /* latent state slot holding x of this chunk          */
  int32_t cond_table;  /* adaLN tables the task reads: its stream id, or
                          max_streams + state_slot for a chunk submitted with
                          its own conditioning (psv_submit_chunk_cond)       */
} psv_task;

/* Per-kernel timing, filled when profiling is on (psv_set_profiling). */
typedef struct psv_kernel_time {
  char    name[32];
  int64_t launches;
  double  total_ms;
  double  flops;       /* algorithmic FLOPs of all launches              */
  double  bytes;       /* algorithmic HBM bytes of all launches          */
} psv_kernel_time;

typedef struct psv_ctx psv_ctx;

/* Device bytes psv_create needs for this description (weights, KV rings
 * for max_streams, activations for the largest wave, latent state, tables):
 * the memory footprint a stream placement checks against (AREX article,
 * section 三层设计, third layer: a stream is admitted only if it fits). */
int psv_arena_bytes(const psv_model_desc* desc, size_t* bytes);

/* Create a context: one served model on one GPU, whose device memory holds
 * the model's weights, every stream's noisy-KV rings and the activations of
 * the largest wave (AREX article, section 三层设计, second layer: one GPU
 * time-shares the stages of many (block, step) pairs and keeps their state).
 * dev_arena/arena_bytes: caller-owned device memory of at
 * least psv_arena_bytes() bytes, 1024-byte aligned, used until psv_destroy;
 * cuda_stream: caller-owned cudaStream_t all device work is issued on
 * (NULL = legacy default stream).  With PSV_FLAG_PLAN_ONLY the arena and
 * stream are ignored (may be NULL) and no CUDA call is made.
 * Errors: PSV_EINVAL (bad shape), PSV_ENOMEM (arena too small), PSV_ECUDA. */
int psv_create(const psv_model_desc* desc, void* dev_arena, size_t arena_bytes,
               void* cuda_stream, psv_ctx** out);

/* Copy n tensors into the arena (see the weight table above).  The model is
 * served as loaded: unpruned, uncompressed, unquantised weights (AREX article,
 * section 实测数字), here bf16 matrices and f32 biases.  Synchronous
 * with respect to the host buffers.  Errors: PSV_EINVAL (unknown id, wrong
 * numel or dtype), PSV_ECUDA. */
int psv_load_weights(psv_ctx* ctx, const psv_weight* w, int n);

/* Open a stream: one agent's sequence of chunks, generated autoregressively
 * and conditioned on that agent (AREX article, section 难题: an
 * action-conditioned world model generates the next frames from the current
 * observation and action; section 三层设计, third layer: each stream is
 * scheduled as a unit).  cond: the stream's conditioning vector (host, f32
 * [d]).  Builds the
 * stream's adaLN tables on the device: for every step s,
 * e_s = T2 SiLU(T1 emb(t_s) + b1) + b2 + cond, mod[s][b] = MOD_W,b SiLU(e_s)
 * + MOD_B,b, fmod[s] = FMOD_W SiLU(e_s) + FMOD_B.  Stream ids are assigned
 * lowest-free-first.  Errors: PSV_EAGAIN (max_streams open), PSV_EINVAL. */
int psv_open_stream(psv_ctx* ctx, const float* cond, int* stream_id);

/* Submit the next chunk of a stream: noise (host, f32 [T, C], the chunk's
 * x_0).  Every chunk starts from pure noise and is denoised over S steps;
 * it may start before its predecessor has finished, reading at each step the
 * predecessor's still-noisy KV of that step (BAAI announcement, section
 * 新一代物理 AI 的基础设施, Fig. 1 right).  Chunks are numbered 0, 1, ... in
 * submission order.  Errors:
 * PSV_EAGAIN (max_inflight chunks alive: poll first), PSV_EINVAL. */
int psv_submit_chunk(psv_ctx* ctx, int stream_id, const float* noise);

/* Submit the next chunk with its own conditioning vector cond (host, f32
 * [d]): an action / observation embedding for this chunk only.  Every step
 * of the chunk uses e_s = temb(t_s) + cond in place of the stream's vector
 * (the pages' action-conditioned world models condition each generated
 * chunk on the agent's action: AREX article, section 难题; BAAI
 * announcement, section 新一代物理 AI 的基础设施).  The chunk's adaLN tables are
 * built on the device before this call returns (asynchronously on the
 * context stream, ahead of any later wave).  Needs a context created with
 * PSV_FLAG_CHUNK_COND.  Errors: PSV_EINVAL (flag missing, null argument),
 * PSV_EAGAIN (max_inflight chunks alive), PSV_ECUDA. */
int psv_submit_chunk_cond(psv_ctx* ctx, int stream_id, const float* noise, const float* cond);

/* Run one wave: every task whose dependencies are met, all streams batched
 * block by block.  The tasks that sit on the same transformer block, from
 * different chunks, denoising steps and streams, run as one batch, so that
 * weight loads and kernel launches are shared (AREX article, section 三层设计,
 * second layer; BAAI announcement, section PhysisServe, time-sharing and
 * Fig. 3 right, cross-stream batching on one card).  Asynchronous on the
 * context stream.  *n_tasks = tasks run (0 = nothing ready; no device work
 * issued). */
int psv_run_wave(psv_ctx* ctx, int* n_tasks);

/* Return the oldest finished, not yet returned chunk of a stream, in chunk
 * order: the stream's output, one chunk per steady interval (BAAI
 * announcement, Fig. 1 right and Fig. 2: once the pipeline is full a new
 * chunk comes out every interval; AREX article, section 实测数字: the output
 * latency is that interval).  Copies
 * its final latent x_S (f32 [T, C]) to host `out` and its index to
 * *chunk_idx.  Non-blocking: PSV_EAGAIN if that chunk's wave has not
 * finished on the device (or no chunk of the stream has been run to its
 * last step).  Checks the device error word: PSV_EDEVICE if set. */
int psv_poll_chunk(psv_ctx* ctx, int stream_id, float* out, int64_t* chunk_idx);

/* Wait (host-side polling, no device spin) until all issued work is done:
 * the end of the time slices issued so far on the one time-shared GPU
 * (AREX article, section 三层设计, second layer).
 * timeout_ms < 0 waits without deadline.  PSV_ETIMEDOUT on deadline. */
int psv_sync(psv_ctx* ctx, int timeout_ms);

/* The task list the next psv_run_wave would run (no state change): the
 * ready (stream, chunk, step) tasks of the dependency DAG of the pages
 * (BAAI announcement, Fig. 2, upper part: one row per stage, one column per
 * chunk).
 * Writes min(n, cap) entries; *n = number of ready tasks. */
int psv_wave_plan(psv_ctx* ctx, psv_task* buf, int cap, int* n);

/* Close a stream; its id and rings become free for a later stream (AREX
 * article, section 三层设计, third layer: streams arrive and leave while
 * others keep running).  Queued work is not
 * cancelled: call after its chunks were polled. */
int psv_close_stream(psv_ctx* ctx, int stream_id);

/* ---- admission control (one GPU) -----------------------------------------
 * The pages admit a new stream only when the whole stream fits and its
 * service objective (SLO) can be met, never migrate running streams, and so
 * keep the service of the streams already admitted stable (AREX article,
 * section 三层设计, third layer; BAAI announcement, section PhysisServe,
 * multi-stream scheduling).  On one GPU: a stream's state is its KV rings
 * (one of the max_streams ring sets reserved at create), and in steady state
 * every open stream gets one chunk per wave, so every stream's ms per chunk
 * is the shared wave time, which a new stream lengthens for all of them.
 *
 * Predicted steady wave time with n open streams (n*S tasks, full windows).
 * The library times every wave on the device and keeps the mean of the
 * full-window waves per task count; a count measured before is predicted by
 * its mean, another one from the nearest measured count in proportion to
 * the algorithmic FLOPs, and with no measurement at all from the
 * algorithmic FLOPs at 1 PFLOP/s.  Errors: PSV_EINVAL (n < 1 or >
 * max_streams). */
int psv_predict_wave_ms(psv_ctx* ctx, int n_streams, double* ms);

/* Open a stream (as psv_open_stream) only if a ring set is free and the
 * predicted wave time with it meets slo_ms (ms per chunk, <= 0: none) and the
 * SLO every open stream was admitted with.  *predicted_ms (may be NULL) gets
 * the prediction.  Errors: PSV_EAGAIN (rejected: no ring set free, or an SLO
 * would be missed; the reason is in psv_last_error), PSV_EINVAL, PSV_ECUDA. */
int psv_admit_stream(psv_ctx* ctx, const float* cond, double slo_ms, int* stream_id,
                     double* predicted_ms);

/* Destroy the context (synchronises the stream first); the arena returns to
 * the caller.  NULL is a no-op.  (Housekeeping: the pages have no
 * counterpart.) */
void psv_destroy(psv_ctx* ctx);

/* Last error message of this context ("" if none); NULL ctx gives the
 * message of the last failed psv_create.  (Housekeeping: the pages have no
 * counterpart.) */
const char* psv_last_error(const psv_ctx* ctx);

/* ---- executor controls and introspection -------------------------------- */

/* Replay each wave shape (task count) as a CUDA graph (default on). */
int psv_set_graphs(psv_ctx* ctx, int enabled);

/* Record CUDA events around every kernel launch (forces eager launches
 * while on).  psv_kernel_times returns per-kernel totals since enabling;
 * it synchronises the stream.  Writes min(cap, kinds) entries, *n = kinds. */
int psv_set_profiling(psv_ctx* ctx, int enabled);
int psv_kernel_times(psv_ctx* ctx, psv_kernel_time* out, int cap, int* n);

/* Debug tap for parity tests: during the next psv_run_wave (run eagerly),
 * copy the residual stream h (f32 [n_tasks*T, d], rows in task order) into
 * the caller's device buffers h_in (before block `block`) and h_out (after
 * it).  Cleared after that wave. */
int psv_debug_tap(psv_ctx* ctx, int block, float* h_in, float* h_out);

/* Debug read of one KV ring (stream, block, step) into host f32 buffers:
 * k [(W+1)*T, d] and v [(W+1)*T, d], rows = slot*T + token.  Synchronous. */
int psv_debug_read_kv(psv_ctx* ctx, int stream_id, int block, int step,
                      float* k, float* v);

/* Debug: byte offset, from the start of the arena given to psv_create, of
 * the int error word that a kernel sets when a device-side wait times out or
 * a bounds check fails (psv_poll_chunk and psv_sync then return the sticky
 * PSV_EDEVICE).  Lets a test raise the word from the host, without any
 * kernel fault, to check that path.  Errors: PSV_EINVAL (plan-only
 * context). */
int psv_debug_error_word(psv_ctx* ctx, size_t* arena_offset);

/* ---- kernel-level window attention ---------------------------------------
 * The attention step of the wave (AREX article "vLLM 与 Physis-AI 联合介绍
 * PhysisServe 推理系统", §难题: a chunk's queries attend to its own keys and
 * the still-noisy keys the preceding chunks left) as a standalone call on
 * caller buffers: n independent query blocks; the T queries of block i
 * attend to the L keys of block i with softmax scale 1/sqrt(dh), no mask.
 *   q   bf16 [n*T][H*dh]            row-major; head h = columns [h*dh, (h+1)*dh)
 *   k   bf16 [n][k_rows][H*dh]      keys of block i at rows [0, L)
 *   vt  bf16 [n][H][dh][vt_cols]    values transposed per head, keys at cols [0, L)
 *   o   bf16 [n*T][H*dh]            output (written)
 * Requirements: dh in {32, 64, 128}; H*dh % 8 == 0; 1 <= L <= k_rows;
 * L <= vt_cols, vt_cols % 8 == 0; all pointers 16-byte aligned device memory.
 * scratch: caller-owned device memory of at least psv_attention_scratch_bytes
 * bytes (task table, the work queue of the persistent CTA pairs and the
 * split-key arrival counters, split-key partials), 256-byte aligned;
 * it is overwritten and must not be shared by calls that may overlap on the
 * GPU.  Asynchronous on cuda_stream; the int at the start of scratch is set
 * nonzero if a device-side pipeline wait timed out.  Errors: PSV_EINVAL. */
typedef struct psv_attn_problem {
  int32_t n, T, H, dh, L, k_rows, vt_cols;
} psv_attn_problem;

int psv_attention_scratch_bytes(const psv_attn_problem* p, size_t* bytes);
int psv_attention(const psv_attn_problem* p, const void* q, const void* k, const void* vt,
                  void* o, void* scratch, size_t scratch_bytes, void* cuda_stream);

/* Allocation-free psv_attention (the pages have no counterpart: this is a
 * deployment convenience).  For callers that cannot allocate device memory
 * at call time, e.g. a real-time control loop that must not enter the CUDA
 * allocator after start-up, or a host framework that owns all device memory
 * and provides no scratch.  Same arguments and results as psv_attention,
 * without scratch: the library uses a fixed array of
 * PSV_ATTN_NOALLOC_SCRATCH_BYTES bytes inside its CUDA module, which every
 * device that loads the module holds until the process exits.  Problems
 * whose scratch (psv_attention_scratch_bytes) exceeds that size are rejected
 * with PSV_ENOMEM; bad shapes or pointers with PSV_EINVAL.
 * Set-up: the first call on a device, with that device current, looks up
 * the array's device address.  Under CUDA's default lazy module loading that
 * is also when the module is loaded on the device and the array reserved, so
 * the first call may fail with PSV_ECUDA if the device is out of memory; make
 * it at start-up, and before any stream capture.  Later calls allocate
 * nothing, on the host or on the device.  Every call shares the one array
 * (each call clears the parts that must start at zero), and the array keeps
 * the last call's contents; calls whose work may overlap on the GPU race on
 * it and must be ordered by the caller (e.g. issued on one stream). */
#define PSV_ATTN_NOALLOC_SCRATCH_BYTES (16u << 20)
int psv_attention_noalloc(const psv_attn_problem* p, const void* q, const void* k,
                          const void* vt, void* o, void* cuda_stream);

/* Status of the last psv_attention_noalloc call on the current device:
 * waits for cuda_stream, then *status = the error word of the shared array
 * (0, or nonzero if a device-side pipeline wait of that call timed out and
 * its output is not valid).  Allocates nothing.  Errors: PSV_EINVAL,
 * PSV_ECUDA. */
int psv_attention_noalloc_status(int* status, void* cuda_stream);

#ifdef __cplusplus
}
#endif

#endif /* PSV_H */
