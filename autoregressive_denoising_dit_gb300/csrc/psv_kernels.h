// Host-visible launch interface of libpsv's kernels (internal to the
// library; the public C ABI is include/psv.h).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

namespace psv {

// Runs the set-up step f (function attributes, occupancy queries) once per
// CUDA device, for the device current at the call: an attribute set on one
// device does not carry over to another.  `done` is the caller's bit mask of
// devices already set up (devices 0..63); one lock serialises every set-up.
inline std::mutex& device_setup_mutex() {
  static std::mutex mu;
  return mu;
}
template <class F>
cudaError_t once_per_device(uint64_t* done, F&& f) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(device_setup_mutex());
  if ((*done >> dev) & 1u) return cudaSuccess;
  e = f(dev);
  if (e == cudaSuccess) *done |= uint64_t{1} << dev;
  return e;
}

struct TaskDev;

// Epilogues of the tcgen05 GEMM  C[M, N] = A[M, K] * W[N, K]^T + bias.
enum GemmEpilogue : int {
  EPI_QKV = 0,    // RoPE on q, k; q -> Q buffer, k -> K ring, v -> V^T ring
  EPI_RESID = 1,  // h += gate[task] * C   (gated residual, f32)
  EPI_GELU = 2,   // u = bf16(GELU_tanh(C))
  EPI_EULER = 3,  // x[task] += dt[task] * C   (velocity head + Euler step)
  EPI_STORE = 4,  // h = C + bias (f32, through TMA stores; the in-projection)
};

struct GemmParams {
  int M, N, K;
  int T, d, dh, H, S, B, C;
  int block;               // transformer block b
  int wz;                  // z coordinate of W in its [z][Npad][K] map
  const TaskDev* tasks;
  const float* bias;       // [N]
  // EPI_QKV
  __nv_bfloat16* q_out;    // [rows][d]
  __nv_bfloat16* k_ring;   // [rings][Lr][d]
  __nv_bfloat16* vt_ring;  // [rings][H][dh][Lp]
  int Lr, Lp;
  int vt_box;              // 1: V^T through TMA stores of 32 x 32 boxes (tmE)
  const float2* rope_local;  // [dh/2][T]   (cos, sin) of i * f_j
  const float2* rope_base;   // [slots][dh/2] (cos, sin) of c*T * f_j
  // EPI_RESID
  float* h;                // [rows][d]
  const float* mod;        // adaLN table base
  int gate_off;            // 2d (gate1) or 5d (gate2)
  // EPI_GELU
  __nv_bfloat16* u;        // [rows][N]
  // EPI_EULER
  float* state;            // [slots][T][C]
  int* err;
};

struct AttnParams {
  int T, d, dh, H, S, Lr, Lp;
  int block;
  int n_tasks;
  const TaskDev* tasks;
  __nv_bfloat16* o;        // [rows][d]
  float scale_log2;        // log2(e) / sqrt(dh)
  // Split-KV partials: per (task, head, 256-row query unit) 2 key halves x
  // 2 CTAs of [dh + 2][128] f32 (O transposed, then m, l).  counters: the
  // work queue (kQueueInts: next piece, pairs done; zero between launches),
  // then one arrival counter per (unit, CTA).
  float* part;
  int* counters;
  int max_pairs;           // query units per (task, head) the partial area is sized for
  int n_pieces;            // work pieces of this launch (attn_pieces)
  int* err;
};

// Key tiles (of 256) from which a (task, head, query unit) is split in two
// key halves (two work pieces, merged through global memory); the split
// depends on the task's kv_len and on the unit being a tail only, so the
// result of a task does not depend on the rest of the wave.  Splitting every
// 7800-key window of the 1.3B wave made the attention 12% slower (twice the
// pieces and a merge), so only windows of 16K keys and more are split.
constexpr int kAttnSplitMinTiles = 64;
// Tail units (the last query unit of a task when its rows fit in one CTA,
// e.g. 24 of T = 1560) cost as much as a full unit; from this many key tiles
// (2K keys) they are split into two halves, short pieces that the work queue
// hands out late so that they even out the end of the launch.
constexpr int kAttnTailSplitMinTiles = 8;
constexpr int kQueueInts = 2;
// Query units of 256 rows per (task, head).
int attn_units(int T);
// Work pieces (256 query rows x a whole window or one key half) of a launch
// over these kv lengths.
int attn_pieces(const int* kv_lens, int n_tasks, int T, int H);
// The same for n tasks that all attend to L keys.
int attn_pieces_uniform(int L, int n_tasks, int T, int H);
// CTAs (two per pair) of a persistent launch: one pair per two SMs at most.
int attn_grid_size(int n_pieces, int sm_count);
size_t attn_part_floats(int max_tasks, int T, int H, int dh);
size_t attn_counter_ints(int max_tasks, int T, int H);
// Each CTA of a pair loads dh/2 rows of a V^T tile: the box height of the
// V^T tensor map.
inline uint32_t attn_v_box_rows(int dh) { return static_cast<uint32_t>(dh / 2); }
// Each CTA of a pair loads 128 keys of a 256-key tile: the box height of the
// K tensor map.
inline uint32_t attn_k_box_rows() { return 128u; }

constexpr int kGemmBM = 128, kGemmBN = 256;  // rows per CTA, columns of the narrow pair tile
size_t gemm_smem_bytes();
size_t attn_smem_bytes(int dh);

// tmC: output map of the epilogues that write through TMA: f32 h ([rows][d],
// box 32 x 32, 128-byte swizzle) for EPI_RESID (TMA reduce-add), bf16 u
// ([rows][F], box 64 x 32, 128-byte swizzle) for EPI_GELU, bf16 q ([rows][d],
// box 64 x 32, 128-byte swizzle) for EPI_QKV; tmD: bf16 K ring ([rings][Lr][d],
// box 64 x 32 x 1, 128-byte swizzle) for EPI_QKV (both needed when d % 64 == 0);
// tmE: bf16 V^T ring ([rings*H][dh][Lp], box 32 x 32 x 1, no swizzle) for
// EPI_QKV when p.vt_box is set.  The others ignore them.
cudaError_t launch_gemm(int epi, const CUtensorMap* tmA, const CUtensorMap* tmB,
                        const CUtensorMap* tmC, const CUtensorMap* tmD, const CUtensorMap* tmE,
                        const GemmParams& p, int grid, cudaStream_t st);
cudaError_t launch_attention(const CUtensorMap* tmQ, const CUtensorMap* tmK,
                             const CUtensorMap* tmV, const AttnParams& p, int n_tasks, int grid,
                             cudaStream_t st);

// Memory-bound kernels.
// y = bf16(LN(h) * (1 + scale) + shift), per row; shift/scale of the row's
// task at mod + task.mod0 + block*6d + {shift_off, scale_off} (or fmod).
// err: the device error word its bounded waits raise (rows of up to 2048
// values are staged by bulk copies; null: the register kernel only).
cudaError_t launch_ln_mod(const float* h, __nv_bfloat16* y, int M, int d, int T,
                          const TaskDev* tasks, const float* table, int use_fmod, int block,
                          int shift_off, int scale_off, float eps, int* err, cudaStream_t st);
// In-projection h = x W_in^T + b_in on the tensor cores: x (f32, gathered
// from each task's latent state slot) is split into bf16 hi + lo parts,
// xs[r] = [hi(x_r) | lo(x_r) | 0...] (K2 columns), so that a bf16 GEMM
// against W2 = [W_in | W_in | 0...] gives x W_in^T with x kept to 2^-16 relative.
cudaError_t launch_in_split(const float* state, const TaskDev* tasks, __nv_bfloat16* xs, int M,
                            int C, int T, int K2, cudaStream_t st);
// W2 [rows][K2] = [W_in | W_in | 0...] from W_in [d][C] (rows >= d: zero).
cudaError_t launch_build_in2(const __nv_bfloat16* w_in, __nv_bfloat16* w_in2, int d, int C,
                             int K2, int rows, cudaStream_t st);
// out[r][n] = act(in[r]) . W[n] + b[n] (+ add[n]), r < R; act = SiLU or id.
cudaError_t launch_cond_linear(const float* in, int R, int K, const __nv_bfloat16* W,
                               const float* b, const float* add, float* out, int N,
                               int silu_in, cudaStream_t st);
cudaError_t launch_f32_to_bf16(const float* src, __nv_bfloat16* dst, int64_t n, cudaStream_t st);
// Task table of a standalone attention call: block i = rows [i*T, i*T+T),
// keys of "ring" i, kv_len = L.
cudaError_t launch_fill_attn_tasks(TaskDev* tasks, int n, int T, int L, cudaStream_t st);

// bf16 tiled tensor map (dims innermost first, strides in bytes for dims
// 1..rank-1); false if the driver entry point or the arguments are rejected.
bool encode_bf16_map(CUtensorMap* map, int rank, void* base, const uint64_t* dims,
                     const uint64_t* strides, const uint32_t* box, CUtensorMapSwizzle sw);
// The same for f32 elements.
bool encode_f32_map(CUtensorMap* map, int rank, void* base, const uint64_t* dims,
                    const uint64_t* strides, const uint32_t* box, CUtensorMapSwizzle sw);

}  // namespace psv
