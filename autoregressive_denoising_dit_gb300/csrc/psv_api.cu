// libpsv host runtime: arena planner, tensor maps, the wave scheduler, the
// wave executor (CUDA-graph replay per wave shape) and the C ABI of psv.h.
//
// Scheduling follows the pages' task DAG (AREX article "vLLM 与 Physis-AI
// 联合介绍 PhysisServe 推理系统", §难题 and §三层设计; BAAI announcement
// "智源悟界·PhysisServe", Fig. 1–3): chunk c step s of a stream is ready when
// chunk c has finished step s-1 and chunk c-1 has finished step s.  Chunks
// finish a step in order, so a stream's whole progress is one counter per
// step: done[s] = chunks that finished step s; step s is ready for chunk
// done[s] when that chunk exists and has finished step s-1.  Every ready task
// of every stream forms one wave, ordered by (stream, step); the wave runs
// block by block with one batched launch per operation (same-block batching,
// Fig. 3 right).
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <chrono>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <map>
#include <string>
#include <thread>
#include <vector>

#include "../../include/psv.h"
#include "psv_device.cuh"
#include "psv_kernels.h"

#define PSV_API extern "C" __attribute__((visibility("default")))

using psv::TaskDev;

namespace {

constexpr size_t kAlign = 1024;
constexpr int kTaskBufs = 16;
constexpr int kWaveEvents = 64;

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
int64_t round_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }

struct Layout {
  // derived sizes
  int Npad_qkv, Npad_o, Npad_up, Npad_down, Npad_out;
  int Lr, Lp, n_rings, n_slots, max_tasks, M_max;
  int n_ctabs;  // conditioning tables: one per stream, plus one per chunk slot with PSV_FLAG_CHUNK_COND
  // byte offsets into the arena
  size_t w_qkv, w_o, w_up, w_down, w_mod;
  size_t b_qkv, b_o, b_up, b_down, b_mod;
  size_t w_in, b_in, w_t1, b_t1, w_t2, b_t2, w_fmod, b_fmod, w_out, b_out;
  size_t w_in2, xs;  // in-projection operands: [W_in | W_in] and [hi(x) | lo(x)], K2 columns
  int K2;
  size_t weights_end;
  size_t k_ring, vt_ring, rings_end;
  size_t h, y, q, o, u, acts_end;
  size_t state, mod, fmod, rope_local, rope_base, tasks, err, scratch;
  size_t temb_in;  // timestep sinusoids of t_0..t_{S-1}, f32 [S][t_embed]
  size_t ccond;    // per-chunk conditioning vectors, f32 [n_slots][d] (PSV_FLAG_CHUNK_COND)
  size_t attn_part, attn_cnt;  // split-KV partials and arrival counters
  int attn_pairs;
  size_t total;
};

int validate(const psv_model_desc* d, std::string* why) {
  auto fail = [&](const char* m) {
    *why = m;
    return PSV_EINVAL;
  };
  if (!d) return fail("null model description");
  if (d->B < 1 || d->S < 1 || d->S > 8) return fail("need B >= 1 and 1 <= S <= 8");
  if (d->d < 128 || d->d % 128 != 0) return fail("d must be a positive multiple of 128");
  if (d->dh != 32 && d->dh != 64 && d->dh != 128) return fail("dh must be 32, 64 or 128");
  if (d->H * d->dh != d->d) return fail("H * dh must equal d");
  if (d->F < 64 || d->F % 64 != 0) return fail("F must be a positive multiple of 64");
  if (d->C < 1 || d->C > 256) return fail("C must be in 1..256");
  if (d->T < 1) return fail("T must be >= 1");
  if (d->W < 0) return fail("W must be >= 0");
  if (d->max_streams < 1) return fail("max_streams must be >= 1");
  if (d->max_inflight < 0) return fail("max_inflight must be >= 0");
  if (d->t_embed < 2 || d->t_embed % 8 != 0 || d->t_embed > 1024)
    return fail("t_embed must be a multiple of 8 in 8..1024");
  if (!(d->ln_eps > 0.0f) || !(d->rope_theta > 1.0f)) return fail("bad ln_eps or rope_theta");
  if (d->d > 6144) return fail("d > 6144 is not supported by the LayerNorm kernel");
  const int64_t rows = static_cast<int64_t>(d->max_streams) * d->S * d->T;
  if (rows > (1 << 30) / 8) return fail("wave too large");
  const int64_t lr = static_cast<int64_t>(d->W + 1) * d->T;
  if (lr > (1 << 28)) return fail("KV window too long");
  // adaLN table offsets are 32-bit float offsets (TaskDev.mod0)
  const int64_t inflight = d->max_inflight > 0 ? d->max_inflight : d->S + 4;
  const int64_t ctabs = d->max_streams + ((d->flags & PSV_FLAG_CHUNK_COND) ? d->max_streams * inflight : 0);
  if (ctabs * d->S * d->B * 6 * static_cast<int64_t>(d->d) >= (int64_t{1} << 31))
    return fail("adaLN tables too large (streams x in-flight chunks x steps x blocks x 6d)");
  return PSV_OK;
}

int inflight_of(const psv_model_desc& d) { return d.max_inflight > 0 ? d.max_inflight : d.S + 4; }

Layout plan_layout(const psv_model_desc& m) {
  Layout L{};
  const int64_t d = m.d, F = m.F, C = m.C, B = m.B, S = m.S;
  L.Npad_qkv = static_cast<int>(round_up(3 * d, 256));
  L.Npad_o = static_cast<int>(round_up(d, 256));
  L.Npad_up = static_cast<int>(round_up(F, 256));
  L.Npad_down = static_cast<int>(round_up(d, 256));
  L.Npad_out = 256;
  L.Lr = (m.W + 1) * m.T;
  L.Lp = static_cast<int>(round_up(L.Lr, 64));
  L.n_rings = m.max_streams * m.B * m.S;
  L.n_slots = m.max_streams * inflight_of(m);
  L.n_ctabs = m.max_streams + ((m.flags & PSV_FLAG_CHUNK_COND) ? L.n_slots : 0);
  L.max_tasks = m.max_streams * m.S;
  L.M_max = static_cast<int>(round_up(static_cast<int64_t>(L.max_tasks) * m.T, 128));
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = align_up(off + bytes, kAlign);
    return at;
  };
  L.w_qkv = take(B * L.Npad_qkv * d * 2);
  L.w_o = take(B * L.Npad_o * d * 2);
  L.w_up = take(B * L.Npad_up * d * 2);
  L.w_down = take(B * L.Npad_down * F * 2);
  L.w_mod = take(B * 6 * d * d * 2);
  L.b_qkv = take(B * 3 * d * 4);
  L.b_o = take(B * d * 4);
  L.b_up = take(B * F * 4);
  L.b_down = take(B * d * 4);
  L.b_mod = take(B * 6 * d * 4);
  L.w_in = take(d * C * 2);
  L.b_in = take(d * 4);
  L.K2 = static_cast<int>(round_up(2 * C, 64));
  L.w_in2 = take(static_cast<size_t>(L.Npad_o) * L.K2 * 2);
  L.w_t1 = take(d * m.t_embed * 2);
  L.b_t1 = take(d * 4);
  L.w_t2 = take(d * d * 2);
  L.b_t2 = take(d * 4);
  L.w_fmod = take(2 * d * d * 2);
  L.b_fmod = take(2 * d * 4);
  L.w_out = take(static_cast<size_t>(L.Npad_out) * d * 2);
  L.b_out = take(256 * 4);
  L.weights_end = off;
  L.k_ring = take(static_cast<size_t>(L.n_rings) * L.Lr * d * 2);
  L.vt_ring = take(static_cast<size_t>(L.n_rings) * d * L.Lp * 2);
  L.rings_end = off;
  L.h = take(static_cast<size_t>(L.M_max) * d * 4);
  L.y = take(static_cast<size_t>(L.M_max) * d * 2);
  L.q = take(static_cast<size_t>(L.M_max) * d * 2);
  L.o = take(static_cast<size_t>(L.M_max) * d * 2);
  L.u = take(static_cast<size_t>(L.M_max) * F * 2);
  L.xs = take(static_cast<size_t>(L.M_max) * L.K2 * 2);
  L.acts_end = off;
  L.state = take(static_cast<size_t>(L.n_slots) * m.T * C * 4);
  L.mod = take(static_cast<size_t>(L.n_ctabs) * S * B * 6 * d * 4);
  L.fmod = take(static_cast<size_t>(L.n_ctabs) * S * 2 * d * 4);
  L.temb_in = take(static_cast<size_t>(S) * m.t_embed * 4);
  L.ccond = take((m.flags & PSV_FLAG_CHUNK_COND) ? static_cast<size_t>(L.n_slots) * d * 4 : 4);
  L.rope_local = take(static_cast<size_t>(m.T) * (m.dh / 2) * 8);
  L.rope_base = take(static_cast<size_t>(L.n_slots) * (m.dh / 2) * 8);
  L.tasks = take(static_cast<size_t>(L.max_tasks) * sizeof(TaskDev));
  L.err = take(256);
  L.scratch = take(static_cast<size_t>(8) * (m.t_embed + 3 * d) * 4 + d * 4);
  L.attn_pairs = psv::attn_units(m.T);
  L.attn_part = take(psv::attn_part_floats(L.max_tasks, m.T, m.H, m.dh) * 4);
  L.attn_cnt = take(psv::attn_counter_ints(L.max_tasks, m.T, m.H) * 4);
  L.total = off;
  return L;
}

PFN_cuTensorMapEncodeTiled_v12000 get_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

}  // namespace

namespace {
bool encode_map(CUtensorMapDataType dt, CUtensorMap* map, int rank, void* base,
                const uint64_t* dims, const uint64_t* strides, const uint32_t* box,
                CUtensorMapSwizzle sw) {
  auto enc = get_encoder();
  if (!enc) return false;
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = enc(map, dt, rank, base, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}
}  // namespace

bool psv::encode_bf16_map(CUtensorMap* map, int rank, void* base, const uint64_t* dims,
                          const uint64_t* strides, const uint32_t* box, CUtensorMapSwizzle sw) {
  return encode_map(CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, map, rank, base, dims, strides, box, sw);
}

bool psv::encode_f32_map(CUtensorMap* map, int rank, void* base, const uint64_t* dims,
                         const uint64_t* strides, const uint32_t* box, CUtensorMapSwizzle sw) {
  return encode_map(CU_TENSOR_MAP_DATA_TYPE_FLOAT32, map, rank, base, dims, strides, box, sw);
}

namespace {

bool encode_bf16(CUtensorMap* map, int rank, void* base, const uint64_t* dims,
                 const uint64_t* strides, const uint32_t* box, CUtensorMapSwizzle sw) {
  return psv::encode_bf16_map(map, rank, base, dims, strides, box, sw);
}

uint16_t f32_to_bf16_bits(float f) {
  uint32_t u;
  std::memcpy(&u, &f, 4);
  if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return static_cast<uint16_t>((u >> 16) | 0x40);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return static_cast<uint16_t>(u >> 16);
}
float bf16_bits_to_f32(uint16_t b) {
  uint32_t u = static_cast<uint32_t>(b) << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return f;
}

enum KernelKind { K_IN_PROJ, K_LN, K_GEMM_QKV, K_ATTN, K_GEMM_O, K_GEMM_UP, K_GEMM_DOWN,
                  K_GEMM_FINAL, K_COUNT };
const char* kKindNames[K_COUNT] = {"in_proj", "ln_mod", "gemm_qkv_rope", "attention",
                                   "gemm_o_resid", "gemm_up_gelu", "gemm_down_resid",
                                   "gemm_final_euler"};

struct StreamState {
  bool open = false;
  int64_t n_sub = 0, n_polled = 0;
  int64_t done[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  std::vector<int64_t> finish_wave;  // per state slot: wave that finished the chunk
  std::vector<char> own_cond;        // per state slot: chunk submitted with its own cond
  double slo_ms = 0.0;               // SLO the stream was admitted with (0: none)
};

// Device-timed waves, for the admission model.
struct WaveTiming {
  cudaEvent_t t0 = nullptr, t1 = nullptr;
  int n_tasks = 0;
  bool full = false;    // every task had a full window (a steady wave)
  bool pending = false;
};
struct WaveStat {
  int64_t count = 0;
  double mean_ms = 0.0;
};

struct ProfRec {
  int kind;
  cudaEvent_t a, b;
  double flops, bytes;
};

}  // namespace

struct psv_ctx {
  psv_model_desc m{};
  Layout L{};
  bool plan_only = false;
  bool sequential = false;
  bool latency = false;
  cudaStream_t stream = nullptr;
  cudaStream_t copy_stream = nullptr;
  cudaStream_t cap_stream = nullptr;  // private stream graphs are captured on
  char* arena = nullptr;
  int sm_count = 148;
  int inflight = 0;
  std::string err;
  int sticky = PSV_OK;
  bool w_loaded[32] = {};
  std::vector<uint8_t> blk_loaded;  // [B][10]
  std::vector<StreamState> streams;
  int64_t wave_id = 0;
  // pinned staging
  TaskDev* h_tasks = nullptr;  // [kTaskBufs][max_tasks]
  cudaEvent_t task_ev[kTaskBufs] = {};
  int task_buf = 0;
  float* h_noise = nullptr;   // [n_slots][T*C]
  float2* h_rope = nullptr;   // [n_slots][dh/2]
  float* h_out = nullptr;     // [T*C]
  float* h_misc = nullptr;    // conditioning staging
  float* h_ccond = nullptr;   // [n_slots][d] per-chunk conditioning staging
  size_t h_misc_bytes = 0;
  cudaEvent_t wave_ev[kWaveEvents] = {};
  WaveTiming wave_tm[kWaveEvents];
  std::map<int, WaveStat> wave_stats;  // task count -> steady wave time
  // tensor maps
  CUtensorMap tmA_y, tmA_o, tmA_u, tmB_qkv, tmB_o, tmB_up, tmB_down, tmB_out, tmQ, tmK, tmV;
  CUtensorMap tmA_xs, tmB_in2;  // in-projection GEMM operands
  CUtensorMap tmC_h;  // f32 h, the target of the gated-residual TMA reductions
  CUtensorMap tmC_u;  // bf16 u, written by the GELU epilogue's TMA stores
  CUtensorMap tmC_q;  // bf16 q and the K ring, written by the QKV epilogue's
  CUtensorMap tmC_k;  // TMA stores (32-row x 64-column boxes)
  CUtensorMap tmC_vt;  // the transposed V ring, 32 x 32 boxes (QKV epilogue)
  bool vt_box = false;
  // executor
  bool use_graphs = true;
  std::map<int64_t, int> shape_seen;
  std::map<int64_t, cudaGraphExec_t> graphs;
  bool profiling = false;
  std::vector<ProfRec> prof;
  std::vector<cudaEvent_t> ev_pool;
  double kind_ms[K_COUNT] = {}, kind_flops[K_COUNT] = {}, kind_bytes[K_COUNT] = {};
  int64_t kind_launches[K_COUNT] = {};
  // debug tap
  int tap_block = -1;
  float* tap_in = nullptr;
  float* tap_out = nullptr;

  template <class T>
  T* at(size_t off) const { return reinterpret_cast<T*>(arena + off); }
};

namespace {

std::string g_create_error;

int set_err(psv_ctx* c, int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  if (c) c->err = buf;
  else g_create_error = buf;
  return code;
}

int cuda_fail(psv_ctx* c, cudaError_t e, const char* what) {
  set_err(c, PSV_ECUDA, "%s: %s", what, cudaGetErrorString(e));
  if (c) c->sticky = PSV_ECUDA;
  return PSV_ECUDA;
}

#define CK(call, what)                                   \
  do {                                                   \
    cudaError_t e_ = (call);                             \
    if (e_ != cudaSuccess) return cuda_fail(ctx, e_, what); \
  } while (0)

int check_ctx(psv_ctx* ctx) {
  if (!ctx) return PSV_EINVAL;
  if (ctx->sticky) return ctx->sticky;
  return PSV_OK;
}

// ------------------------------------------------------------- scheduling

// Ready tasks of the current state in (stream, step) order (closed form of
// the DAG readiness, see the file header).
void plan_wave(const psv_ctx* ctx, std::vector<psv_task>* out) {
  out->clear();
  const psv_model_desc& m = ctx->m;
  for (int sid = 0; sid < static_cast<int>(ctx->streams.size()); ++sid) {
    const StreamState& st = ctx->streams[sid];
    if (!st.open) continue;
    for (int s = 0; s < m.S; ++s) {
      const int64_t c = st.done[s];
      if (c >= st.n_sub) continue;
      if (s > 0 && st.done[s - 1] <= c) continue;
      psv_task t{};
      t.stream = sid;
      t.chunk = static_cast<int32_t>(c);
      t.step = s;
      t.slot = static_cast<int32_t>(c % (m.W + 1));
      t.kv_len = static_cast<int32_t>((std::min<int64_t>(c, m.W) + 1) * m.T);
      t.state_slot = sid * ctx->inflight + static_cast<int32_t>(c % ctx->inflight);
      t.cond_table = st.own_cond[static_cast<size_t>(c % ctx->inflight)] ? m.max_streams + t.state_slot : sid;
      out->push_back(t);
    }
  }
  if (ctx->latency && !out->empty()) {
    // Latency mode: each stream's oldest ready chunk only (tasks are grouped
    // by stream, steps ascending; the oldest chunk has the lowest index).
    std::vector<psv_task> keep;
    for (const psv_task& t : *out) {
      if (!keep.empty() && keep.back().stream == t.stream) {
        if (t.chunk < keep.back().chunk) keep.back() = t;
      } else {
        keep.push_back(t);
      }
    }
    out->swap(keep);
  }
  if (ctx->sequential && out->size() > 1) {
    auto best = std::min_element(out->begin(), out->end(), [](const psv_task& a, const psv_task& b) {
      if (a.stream != b.stream) return a.stream < b.stream;
      if (a.chunk != b.chunk) return a.chunk < b.chunk;
      return a.step < b.step;
    });
    psv_task keep = *best;
    out->assign(1, keep);
  }
  for (size_t i = 0; i < out->size(); ++i) (*out)[i].row_off = static_cast<int32_t>(i * m.T);
}

TaskDev to_dev(const psv_ctx* ctx, const psv_task& t) {
  const psv_model_desc& m = ctx->m;
  TaskDev d{};
  d.sid = t.stream;
  d.c = t.chunk;
  d.s = t.step;
  d.row0 = t.row_off;
  d.state_slot = t.state_slot;
  d.ring0 = t.stream * m.B * m.S + t.step;
  d.slot = t.slot;
  d.kv_len = t.kv_len;
  d.mod0 = (t.cond_table * m.S + t.step) * m.B * 6 * m.d;
  d.fmod0 = (t.cond_table * m.S + t.step) * 2 * m.d;
  const double ts = 1.0 - static_cast<double>(t.step) / m.S;
  const double tn = 1.0 - static_cast<double>(t.step + 1) / m.S;
  d.dt = static_cast<float>(tn - ts);
  d.rope_slot = t.state_slot;
  return d;
}

// ------------------------------------------------------------- executor

struct Launcher {
  psv_ctx* ctx;
  bool prof;
  cudaStream_t st;
  cudaError_t err = cudaSuccess;
  cudaEvent_t next_event() {
    if (ctx->ev_pool.empty()) {
      cudaEvent_t e;
      cudaEventCreate(&e);
      return e;
    }
    cudaEvent_t e = ctx->ev_pool.back();
    ctx->ev_pool.pop_back();
    return e;
  }
  template <class F>
  void run(int kind, double flops, double bytes, F&& f) {
    if (err != cudaSuccess) return;
    if (prof) {
      ProfRec r{kind, next_event(), next_event(), flops, bytes};
      cudaEventRecord(r.a, st);
      err = f();
      cudaEventRecord(r.b, st);
      ctx->prof.push_back(r);
    } else {
      err = f();
    }
  }
};

psv::GemmParams base_gemm(const psv_ctx* ctx, int M) {
  const psv_model_desc& m = ctx->m;
  psv::GemmParams p{};
  p.M = M;
  p.T = m.T;
  p.d = m.d;
  p.dh = m.dh;
  p.H = m.H;
  p.S = m.S;
  p.B = m.B;
  p.C = m.C;
  p.tasks = ctx->at<TaskDev>(ctx->L.tasks);
  p.err = ctx->at<int>(ctx->L.err);
  p.Lr = ctx->L.Lr;
  p.Lp = ctx->L.Lp;
  return p;
}

// CTAs of a GEMM launch: two per 256-row pair tile (the two CTAs of a pair
// take the two 128-row halves), at most one per SM.
int gemm_grid(const psv_ctx* ctx, int M, int N) {
  const int m_pairs = ((M + psv::kGemmBM - 1) / psv::kGemmBM + 1) / 2;
  const int tiles = m_pairs * ((N + psv::kGemmBN - 1) / psv::kGemmBN);
  return std::max(2, std::min(2 * tiles, ctx->sm_count));
}

// Enqueue every kernel of one wave of n tasks (task table already on the
// device).  `tap` enables the debug copies of h around one block.
cudaError_t enqueue_wave(psv_ctx* ctx, cudaStream_t st, int n, bool prof, bool tap,
                         const std::vector<TaskDev>* host_tasks) {
  const psv_model_desc& m = ctx->m;
  const Layout& L = ctx->L;
  const int M = n * m.T;
  const int d = m.d, F = m.F;
  const TaskDev* tasks = ctx->at<TaskDev>(L.tasks);
  Launcher run{ctx, prof, st};
  const double Md = static_cast<double>(M) * d;

  // In-projection on the tensor cores: split x into bf16 hi + lo, then
  // h = [hi | lo] [W_in | W_in]^T + b_in, stored in f32.
  run.run(K_IN_PROJ, 0.0, M * m.C * 4.0 + static_cast<double>(M) * L.K2 * 2, [&] {
    return psv::launch_in_split(ctx->at<float>(L.state), tasks, ctx->at<__nv_bfloat16>(L.xs), M, m.C,
                                m.T, L.K2, st);
  });
  {
    psv::GemmParams p = base_gemm(ctx, M);
    p.N = d;
    p.K = L.K2;
    p.block = 0;
    p.wz = 0;
    p.bias = ctx->at<float>(L.b_in);
    run.run(K_IN_PROJ, 2.0 * M * m.C * d, static_cast<double>(M) * L.K2 * 2 + static_cast<double>(M) * d * 4, [&] {
      return psv::launch_gemm(psv::EPI_STORE, &ctx->tmA_xs, &ctx->tmB_in2, &ctx->tmC_h, nullptr, nullptr, p,
                              gemm_grid(ctx, M, p.N), st);
    });
  }

  double attn_flops = 0.0, attn_bytes = 0.0;
  std::vector<int> kv_lens;
  for (const TaskDev& t : *host_tasks) {
    attn_flops += 4.0 * m.T * static_cast<double>(t.kv_len) * d;
    attn_bytes += (2.0 * m.T * d + 2.0 * static_cast<double>(t.kv_len) * d) * 2.0;
    kv_lens.push_back(t.kv_len);
  }
  const int attn_pieces = psv::attn_pieces(kv_lens.data(), n, m.T, m.H);
  const int attn_grid = psv::attn_grid_size(attn_pieces, ctx->sm_count);

  for (int b = 0; b < m.B; ++b) {
    if (tap && b == ctx->tap_block && run.err == cudaSuccess)
      run.err = cudaMemcpyAsync(ctx->tap_in, ctx->at<float>(L.h), Md * 4, cudaMemcpyDeviceToDevice, st);
    // LN1 + modulation
    run.run(K_LN, 0, Md * 6.0, [&] {
      return psv::launch_ln_mod(ctx->at<float>(L.h), ctx->at<__nv_bfloat16>(L.y), M, d, m.T, tasks,
                                ctx->at<float>(L.mod), 0, b, 0, d, m.ln_eps, ctx->at<int>(L.err), st);
    });
    // QKV + RoPE + KV append
    {
      psv::GemmParams p = base_gemm(ctx, M);
      p.N = 3 * d;
      p.K = d;
      p.block = b;
      p.wz = b;
      p.bias = ctx->at<float>(L.b_qkv) + static_cast<size_t>(b) * 3 * d;
      p.q_out = ctx->at<__nv_bfloat16>(L.q);
      p.k_ring = ctx->at<__nv_bfloat16>(L.k_ring);
      p.vt_ring = ctx->at<__nv_bfloat16>(L.vt_ring);
      p.rope_local = ctx->at<float2>(L.rope_local);
      p.rope_base = ctx->at<float2>(L.rope_base);
      p.vt_box = ctx->vt_box ? 1 : 0;
      run.run(K_GEMM_QKV, 2.0 * Md * 3 * d, Md * 2 + 3.0 * d * d * 2 + 3 * Md * 2, [&] {
        return psv::launch_gemm(psv::EPI_QKV, &ctx->tmA_y, &ctx->tmB_qkv, &ctx->tmC_q, &ctx->tmC_k,
                                ctx->vt_box ? &ctx->tmC_vt : nullptr, p, gemm_grid(ctx, M, p.N), st);
      });
    }
    // window attention
    {
      psv::AttnParams a{};
      a.T = m.T;
      a.d = d;
      a.dh = m.dh;
      a.H = m.H;
      a.S = m.S;
      a.Lr = L.Lr;
      a.Lp = L.Lp;
      a.block = b;
      a.n_tasks = n;
      a.tasks = tasks;
      a.o = ctx->at<__nv_bfloat16>(L.o);
      a.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(m.dh)));
      a.part = ctx->at<float>(L.attn_part);
      a.counters = ctx->at<int>(L.attn_cnt);
      a.max_pairs = L.attn_pairs;
      a.n_pieces = attn_pieces;
      a.err = ctx->at<int>(L.err);
      run.run(K_ATTN, attn_flops, attn_bytes, [&] {
        return psv::launch_attention(&ctx->tmQ, &ctx->tmK, &ctx->tmV, a, n, attn_grid, st);
      });
    }
    // out-proj + gated residual (gate1)
    {
      psv::GemmParams p = base_gemm(ctx, M);
      p.N = d;
      p.K = d;
      p.block = b;
      p.wz = b;
      p.bias = ctx->at<float>(L.b_o) + static_cast<size_t>(b) * d;
      p.h = ctx->at<float>(L.h);
      p.mod = ctx->at<float>(L.mod);
      p.gate_off = 2 * d;
      run.run(K_GEMM_O, 2.0 * Md * d, Md * 2 + 1.0 * d * d * 2 + Md * 8, [&] {
        return psv::launch_gemm(psv::EPI_RESID, &ctx->tmA_o, &ctx->tmB_o, &ctx->tmC_h, nullptr, nullptr, p, gemm_grid(ctx, M, p.N), st);
      });
    }
    // LN2 + modulation
    run.run(K_LN, 0, Md * 6.0, [&] {
      return psv::launch_ln_mod(ctx->at<float>(L.h), ctx->at<__nv_bfloat16>(L.y), M, d, m.T, tasks,
                                ctx->at<float>(L.mod), 0, b, 3 * d, 4 * d, m.ln_eps, ctx->at<int>(L.err), st);
    });
    // up + GELU
    {
      psv::GemmParams p = base_gemm(ctx, M);
      p.N = F;
      p.K = d;
      p.block = b;
      p.wz = b;
      p.bias = ctx->at<float>(L.b_up) + static_cast<size_t>(b) * F;
      p.u = ctx->at<__nv_bfloat16>(L.u);
      run.run(K_GEMM_UP, 2.0 * Md * F, Md * 2 + 1.0 * F * d * 2 + static_cast<double>(M) * F * 2, [&] {
        return psv::launch_gemm(psv::EPI_GELU, &ctx->tmA_y, &ctx->tmB_up, &ctx->tmC_u, nullptr, nullptr, p, gemm_grid(ctx, M, p.N), st);
      });
    }
    // down + gated residual (gate2)
    {
      psv::GemmParams p = base_gemm(ctx, M);
      p.N = d;
      p.K = F;
      p.block = b;
      p.wz = b;
      p.bias = ctx->at<float>(L.b_down) + static_cast<size_t>(b) * d;
      p.h = ctx->at<float>(L.h);
      p.mod = ctx->at<float>(L.mod);
      p.gate_off = 5 * d;
      run.run(K_GEMM_DOWN, 2.0 * Md * F, static_cast<double>(M) * F * 2 + 1.0 * F * d * 2 + Md * 8, [&] {
        return psv::launch_gemm(psv::EPI_RESID, &ctx->tmA_u, &ctx->tmB_down, &ctx->tmC_h, nullptr, nullptr, p, gemm_grid(ctx, M, p.N), st);
      });
    }
    if (tap && b == ctx->tap_block && run.err == cudaSuccess)
      run.err = cudaMemcpyAsync(ctx->tap_out, ctx->at<float>(L.h), Md * 4, cudaMemcpyDeviceToDevice, st);
  }
  // final adaLN + velocity head + Euler update
  run.run(K_LN, 0, Md * 6.0, [&] {
    return psv::launch_ln_mod(ctx->at<float>(L.h), ctx->at<__nv_bfloat16>(L.y), M, d, m.T, tasks,
                              ctx->at<float>(L.fmod), 1, 0, 0, d, m.ln_eps, ctx->at<int>(L.err), st);
  });
  {
    psv::GemmParams p = base_gemm(ctx, M);
    p.N = m.C;
    p.K = d;
    p.block = 0;
    p.wz = 0;
    p.bias = ctx->at<float>(L.b_out);
    p.state = ctx->at<float>(L.state);
    run.run(K_GEMM_FINAL, 2.0 * Md * m.C, Md * 2 + static_cast<double>(M) * m.C * 8, [&] {
      return psv::launch_gemm(psv::EPI_EULER, &ctx->tmA_y, &ctx->tmB_out, nullptr, nullptr, nullptr, p, gemm_grid(ctx, M, p.N), st);
    });
  }
  return run.err;
}

int collect_profile(psv_ctx* ctx) {
  if (ctx->prof.empty()) return PSV_OK;
  CK(cudaStreamSynchronize(ctx->stream), "profile sync");
  for (ProfRec& r : ctx->prof) {
    float ms = 0.0f;
    cudaEventElapsedTime(&ms, r.a, r.b);
    ctx->kind_ms[r.kind] += ms;
    ctx->kind_flops[r.kind] += r.flops;
    ctx->kind_bytes[r.kind] += r.bytes;
    ctx->kind_launches[r.kind] += 1;
    ctx->ev_pool.push_back(r.a);
    ctx->ev_pool.push_back(r.b);
  }
  ctx->prof.clear();
  return PSV_OK;
}

int read_device_error(psv_ctx* ctx) {
  int v = 0;
  CK(cudaMemcpyAsync(&v, ctx->at<int>(ctx->L.err), sizeof(int), cudaMemcpyDeviceToHost, ctx->copy_stream),
     "error word read");
  CK(cudaStreamSynchronize(ctx->copy_stream), "error word sync");
  if (v != 0) {
    ctx->sticky = PSV_EDEVICE;
    return set_err(ctx, PSV_EDEVICE, "device error word set: %d (%s)", v,
                   v == psv::ERR_GEMM_TIMEOUT ? "GEMM pipeline wait timed out"
                   : v == psv::ERR_ATTN_TIMEOUT ? "attention pipeline wait timed out"
                   : v == psv::ERR_LN_TIMEOUT   ? "LayerNorm row copy wait timed out"
                                                : "bounds check");
  }
  return PSV_OK;
}

}  // namespace

// ======================================================================= ABI

PSV_API int psv_arena_bytes(const psv_model_desc* desc, size_t* bytes) {
  std::string why;
  if (!bytes) return PSV_EINVAL;
  if (int r = validate(desc, &why)) return set_err(nullptr, r, "%s", why.c_str());
  *bytes = plan_layout(*desc).total;
  return PSV_OK;
}

PSV_API int psv_create(const psv_model_desc* desc, void* dev_arena, size_t arena_bytes,
                       void* cuda_stream, psv_ctx** out) {
  std::string why;
  if (!out) return set_err(nullptr, PSV_EINVAL, "null out pointer");
  *out = nullptr;
  if (int r = validate(desc, &why)) return set_err(nullptr, r, "%s", why.c_str());
  psv_ctx* ctx = new psv_ctx();
  ctx->m = *desc;
  ctx->L = plan_layout(*desc);
  ctx->inflight = inflight_of(*desc);
  ctx->plan_only = (desc->flags & PSV_FLAG_PLAN_ONLY) != 0;
  ctx->sequential = (desc->flags & PSV_FLAG_SEQUENTIAL) != 0;
  ctx->latency = (desc->flags & PSV_FLAG_LATENCY) != 0;
  ctx->blk_loaded.assign(static_cast<size_t>(desc->B) * 16, 0);
  ctx->streams.resize(desc->max_streams);
  for (auto& s : ctx->streams) s.finish_wave.assign(ctx->inflight, -1);
  if (ctx->plan_only) {
    *out = ctx;
    return PSV_OK;
  }
  auto bail = [&](int code) {
    g_create_error = ctx->err;
    psv_destroy(ctx);
    return code;
  };
  if (!dev_arena) { set_err(ctx, PSV_EINVAL, "null arena"); return bail(PSV_EINVAL); }
  if (reinterpret_cast<uintptr_t>(dev_arena) % kAlign) {
    set_err(ctx, PSV_EINVAL, "arena must be 1024-byte aligned");
    return bail(PSV_EINVAL);
  }
  if (arena_bytes < ctx->L.total) {
    set_err(ctx, PSV_ENOMEM, "arena too small: %zu < %zu bytes", arena_bytes, ctx->L.total);
    return bail(PSV_ENOMEM);
  }
  ctx->arena = static_cast<char*>(dev_arena);
  ctx->stream = static_cast<cudaStream_t>(cuda_stream);
  const Layout& L = ctx->L;
  const psv_model_desc& m = ctx->m;
  cudaError_t e;
  int dev = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) { cuda_fail(ctx, e, "cudaGetDevice"); return bail(PSV_ECUDA); }
  cudaDeviceGetAttribute(&ctx->sm_count, cudaDevAttrMultiProcessorCount, dev);
  int cc_major = 0, cc_minor = 0;
  cudaDeviceGetAttribute(&cc_major, cudaDevAttrComputeCapabilityMajor, dev);
  cudaDeviceGetAttribute(&cc_minor, cudaDevAttrComputeCapabilityMinor, dev);
  if (cc_major != 10 || cc_minor != 3) {
    set_err(ctx, PSV_EINVAL, "libpsv is built for sm_103a; device is sm_%d%d", cc_major, cc_minor);
    return bail(PSV_EINVAL);
  }
  if ((e = cudaStreamCreateWithFlags(&ctx->copy_stream, cudaStreamNonBlocking)) != cudaSuccess ||
      (e = cudaStreamCreateWithFlags(&ctx->cap_stream, cudaStreamNonBlocking)) != cudaSuccess) {
    cuda_fail(ctx, e, "copy stream");
    return bail(PSV_ECUDA);
  }
  const size_t tc = static_cast<size_t>(m.T) * m.C;
  ctx->h_misc_bytes = static_cast<size_t>(8) * m.t_embed * 4 + static_cast<size_t>(m.d) * 4;
  if (cudaMallocHost(&ctx->h_tasks, sizeof(TaskDev) * L.max_tasks * kTaskBufs) != cudaSuccess ||
      cudaMallocHost(&ctx->h_noise, tc * 4 * L.n_slots) != cudaSuccess ||
      cudaMallocHost(&ctx->h_rope, static_cast<size_t>(L.n_slots) * (m.dh / 2) * 8) != cudaSuccess ||
      cudaMallocHost(&ctx->h_out, tc * 4) != cudaSuccess ||
      cudaMallocHost(&ctx->h_misc, ctx->h_misc_bytes) != cudaSuccess ||
      ((m.flags & PSV_FLAG_CHUNK_COND) &&
       cudaMallocHost(&ctx->h_ccond, static_cast<size_t>(L.n_slots) * m.d * 4) != cudaSuccess)) {
    set_err(ctx, PSV_ENOMEM, "pinned host staging allocation failed");
    return bail(PSV_ENOMEM);
  }
  for (int i = 0; i < kTaskBufs; ++i) cudaEventCreateWithFlags(&ctx->task_ev[i], cudaEventDisableTiming);
  for (int i = 0; i < kWaveEvents; ++i) {
    cudaEventCreateWithFlags(&ctx->wave_ev[i], cudaEventDisableTiming);
    cudaEventCreate(&ctx->wave_tm[i].t0);
    cudaEventCreate(&ctx->wave_tm[i].t1);
  }
  // Zero the whole arena: padded weight rows, rings (masked keys must be
  // finite), activations, tables and the error word.
  if ((e = cudaMemsetAsync(ctx->arena, 0, L.total, ctx->stream)) != cudaSuccess) {
    cuda_fail(ctx, e, "arena clear");
    return bail(PSV_ECUDA);
  }
  // Timestep sinusoids of t_s = 1 - s/S, in f64: [cos(t f_j), sin(t f_j)],
  // f_j = exp(-ln(1e4) j / (E/2)); shared by every stream and chunk table.
  {
    const int E = m.t_embed;
    std::vector<float> emb(static_cast<size_t>(m.S) * E);
    for (int s = 0; s < m.S; ++s) {
      const double t = 1.0 - static_cast<double>(s) / m.S;
      for (int j = 0; j < E / 2; ++j) {
        const double f = std::exp(-std::log(1e4) * j / (E / 2));
        emb[static_cast<size_t>(s) * E + j] = static_cast<float>(std::cos(t * f));
        emb[static_cast<size_t>(s) * E + E / 2 + j] = static_cast<float>(std::sin(t * f));
      }
    }
    if ((e = cudaMemcpyAsync(ctx->at<float>(L.temb_in), emb.data(), emb.size() * 4, cudaMemcpyHostToDevice,
                             ctx->stream)) != cudaSuccess ||
        (e = cudaStreamSynchronize(ctx->stream)) != cudaSuccess) {
      cuda_fail(ctx, e, "timestep table upload");
      return bail(PSV_ECUDA);
    }
  }
  // RoPE table of in-chunk offsets: (cos, sin) of i * theta^(-2j/dh), f64.
  {
    // stored [dh/2][T] so that the QKV epilogue's per-row reads coalesce
    std::vector<float2> tab(static_cast<size_t>(m.T) * (m.dh / 2));
    for (int i = 0; i < m.T; ++i)
      for (int j = 0; j < m.dh / 2; ++j) {
        const double ang = static_cast<double>(i) * std::pow(static_cast<double>(m.rope_theta), -2.0 * j / m.dh);
        tab[static_cast<size_t>(j) * m.T + i] = make_float2(static_cast<float>(std::cos(ang)),
                                                            static_cast<float>(std::sin(ang)));
      }
    if ((e = cudaMemcpy(ctx->at<float2>(L.rope_local), tab.data(), tab.size() * 8, cudaMemcpyHostToDevice)) !=
        cudaSuccess) {
      cuda_fail(ctx, e, "rope table upload");
      return bail(PSV_ECUDA);
    }
  }
  // Tensor maps (all addresses are fixed for the context's lifetime).
  {
    const uint64_t d = m.d, F = m.F, Mx = L.M_max;
    bool ok = true;
    const CUtensorMapSwizzle SW128 = CU_TENSOR_MAP_SWIZZLE_128B;
    {
      uint64_t dims[2] = {d, Mx}, str[1] = {d * 2};
      uint32_t box[2] = {64, 128};
      ok &= encode_bf16(&ctx->tmA_y, 2, ctx->arena + L.y, dims, str, box, SW128);
      ok &= encode_bf16(&ctx->tmA_o, 2, ctx->arena + L.o, dims, str, box, SW128);
    }
    {
      uint64_t dims[2] = {static_cast<uint64_t>(L.K2), Mx}, str[1] = {static_cast<uint64_t>(L.K2) * 2};
      uint32_t box[2] = {64, 128};
      ok &= encode_bf16(&ctx->tmA_xs, 2, ctx->arena + L.xs, dims, str, box, SW128);
    }
    {
      uint64_t dims[2] = {F, Mx}, str[1] = {F * 2};
      uint32_t box[2] = {64, 128};
      ok &= encode_bf16(&ctx->tmA_u, 2, ctx->arena + L.u, dims, str, box, SW128);
      uint32_t obox[2] = {64, 32};
      ok &= encode_bf16(&ctx->tmC_u, 2, ctx->arena + L.u, dims, str, obox, SW128);
    }
    {
      // h as the target of 32 x 32 f32 boxes (128-byte rows, swizzled)
      uint64_t dims[2] = {d, Mx}, str[1] = {d * 4};
      uint32_t box[2] = {32, 32};
      ok &= psv::encode_f32_map(&ctx->tmC_h, 2, ctx->arena + L.h, dims, str, box, SW128);
    }
    // weight tiles are loaded as two 128-row halves (one per CTA of a cluster)
    auto wmap = [&](CUtensorMap* mp, size_t off, uint64_t K, uint64_t Np, uint64_t Z) {
      uint64_t dims[3] = {K, Np, Z}, str[2] = {K * 2, K * Np * 2};
      uint32_t box[3] = {64, 128, 1};
      return encode_bf16(mp, 3, ctx->arena + off, dims, str, box, SW128);
    };
    ok &= wmap(&ctx->tmB_qkv, L.w_qkv, d, L.Npad_qkv, m.B);
    ok &= wmap(&ctx->tmB_o, L.w_o, d, L.Npad_o, m.B);
    ok &= wmap(&ctx->tmB_up, L.w_up, d, L.Npad_up, m.B);
    ok &= wmap(&ctx->tmB_down, L.w_down, F, L.Npad_down, m.B);
    ok &= wmap(&ctx->tmB_out, L.w_out, d, L.Npad_out, 1);
    ok &= wmap(&ctx->tmB_in2, L.w_in2, L.K2, L.Npad_o, 1);
    const uint32_t aw = m.dh < 64 ? m.dh : 64;
    const CUtensorMapSwizzle swq = aw == 32 ? CU_TENSOR_MAP_SWIZZLE_64B : SW128;
    {
      uint64_t dims[2] = {d, Mx}, str[1] = {d * 2};
      uint32_t box[2] = {aw, 128};
      ok &= encode_bf16(&ctx->tmQ, 2, ctx->arena + L.q, dims, str, box, swq);
    }
    {
      uint64_t dims[3] = {d, static_cast<uint64_t>(L.Lr), static_cast<uint64_t>(L.n_rings)};
      uint64_t str[2] = {d * 2, d * 2 * L.Lr};
      uint32_t box[3] = {aw, psv::attn_k_box_rows(), 1};
      ok &= encode_bf16(&ctx->tmK, 3, ctx->arena + L.k_ring, dims, str, box, swq);
      if (d % 64 == 0) {
        uint32_t obox[3] = {64, 32, 1};
        ok &= encode_bf16(&ctx->tmC_k, 3, ctx->arena + L.k_ring, dims, str, obox, SW128);
        uint64_t qdims[2] = {d, Mx}, qstr[1] = {d * 2};
        uint32_t qbox[2] = {64, 32};
        ok &= encode_bf16(&ctx->tmC_q, 2, ctx->arena + L.q, qdims, qstr, qbox, SW128);
      }
    }
    {
      uint64_t dims[3] = {static_cast<uint64_t>(L.Lp), static_cast<uint64_t>(m.dh),
                          static_cast<uint64_t>(L.n_rings) * m.H};
      uint64_t str[2] = {static_cast<uint64_t>(L.Lp) * 2, static_cast<uint64_t>(L.Lp) * 2 * m.dh};
      uint32_t box[3] = {64, psv::attn_v_box_rows(m.dh), 1};
      ok &= encode_bf16(&ctx->tmV, 3, ctx->arena + L.vt_ring, dims, str, box, SW128);
      // V^T boxes of 32 tokens x 32 dims, stored by the QKV epilogue: their
      // first token (a ring row) must be 8-aligned, so T % 8 == 0
      ctx->vt_box = m.T % 8 == 0 && m.dh % 32 == 0;
      if (ctx->vt_box) {
        uint32_t vbox[3] = {32, 32, 1};
        ok &= encode_bf16(&ctx->tmC_vt, 3, ctx->arena + L.vt_ring, dims, str, vbox,
                          CU_TENSOR_MAP_SWIZZLE_NONE);
      }
    }
    if (!ok) {
      set_err(ctx, PSV_ECUDA, "cuTensorMapEncodeTiled failed (driver entry point or arguments)");
      ctx->sticky = PSV_ECUDA;
      return bail(PSV_ECUDA);
    }
  }
  if ((e = cudaStreamSynchronize(ctx->stream)) != cudaSuccess) {
    cuda_fail(ctx, e, "create sync");
    return bail(PSV_ECUDA);
  }
  *out = ctx;
  return PSV_OK;
}

PSV_API int psv_load_weights(psv_ctx* ctx, const psv_weight* w, int n) {
  if (int r = check_ctx(ctx)) return r;
  if (n < 0 || (n > 0 && !w)) return set_err(ctx, PSV_EINVAL, "bad weight list");
  const psv_model_desc& m = ctx->m;
  const Layout& L = ctx->L;
  const int64_t d = m.d, F = m.F, C = m.C;
  for (int i = 0; i < n; ++i) {
    const psv_weight& x = w[i];
    int64_t numel = -1;
    size_t off = 0;
    bool matrix = false;
    const bool global = x.block < 0;
    if (!global && x.block >= m.B) return set_err(ctx, PSV_EINVAL, "weight %d: block %d out of range", i, x.block);
    const int64_t b = global ? 0 : x.block;
    switch (x.id) {
      case PSV_W_IN_W: numel = d * C; off = L.w_in; matrix = true; break;
      case PSV_W_IN_B: numel = d; off = L.b_in; break;
      case PSV_W_T1_W: numel = d * m.t_embed; off = L.w_t1; matrix = true; break;
      case PSV_W_T1_B: numel = d; off = L.b_t1; break;
      case PSV_W_T2_W: numel = d * d; off = L.w_t2; matrix = true; break;
      case PSV_W_T2_B: numel = d; off = L.b_t2; break;
      case PSV_W_FMOD_W: numel = 2 * d * d; off = L.w_fmod; matrix = true; break;
      case PSV_W_FMOD_B: numel = 2 * d; off = L.b_fmod; break;
      case PSV_W_OUT_W: numel = C * d; off = L.w_out; matrix = true; break;
      case PSV_W_OUT_B: numel = C; off = L.b_out; break;
      case PSV_W_QKV_W: numel = 3 * d * d; off = L.w_qkv + b * L.Npad_qkv * d * 2; matrix = true; break;
      case PSV_W_QKV_B: numel = 3 * d; off = L.b_qkv + b * 3 * d * 4; break;
      case PSV_W_O_W: numel = d * d; off = L.w_o + b * L.Npad_o * d * 2; matrix = true; break;
      case PSV_W_O_B: numel = d; off = L.b_o + b * d * 4; break;
      case PSV_W_UP_W: numel = F * d; off = L.w_up + b * L.Npad_up * d * 2; matrix = true; break;
      case PSV_W_UP_B: numel = F; off = L.b_up + b * F * 4; break;
      case PSV_W_DOWN_W: numel = d * F; off = L.w_down + b * L.Npad_down * F * 2; matrix = true; break;
      case PSV_W_DOWN_B: numel = d; off = L.b_down + b * d * 4; break;
      case PSV_W_MOD_W: numel = 6 * d * d; off = L.w_mod + b * 6 * d * d * 2; matrix = true; break;
      case PSV_W_MOD_B: numel = 6 * d; off = L.b_mod + b * 6 * d * 4; break;
      default: return set_err(ctx, PSV_EINVAL, "weight %d: unknown id %d", i, x.id);
    }
    const bool is_block_id = x.id >= PSV_W_QKV_W;
    if (is_block_id == global)
      return set_err(ctx, PSV_EINVAL, "weight %d: id %d %s a block index", i, x.id, global ? "needs" : "takes no");
    if (x.numel != numel) return set_err(ctx, PSV_EINVAL, "weight %d: numel %lld, expected %lld", i,
                                         static_cast<long long>(x.numel), static_cast<long long>(numel));
    if (!x.data) return set_err(ctx, PSV_EINVAL, "weight %d: null data", i);
    if (x.dtype != PSV_DTYPE_F32 && x.dtype != PSV_DTYPE_BF16) return set_err(ctx, PSV_EINVAL, "weight %d: bad dtype", i);
    if (ctx->plan_only) continue;
    char* dst = ctx->arena + off;
    if (x.location == PSV_LOC_DEVICE) {
      if (matrix && x.dtype == PSV_DTYPE_BF16) {
        CK(cudaMemcpyAsync(dst, x.data, numel * 2, cudaMemcpyDeviceToDevice, ctx->stream), "weight copy");
      } else if (matrix) {
        CK(psv::launch_f32_to_bf16(static_cast<const float*>(x.data), reinterpret_cast<__nv_bfloat16*>(dst), numel,
                                   ctx->stream), "weight cast");
      } else if (x.dtype == PSV_DTYPE_F32) {
        CK(cudaMemcpyAsync(dst, x.data, numel * 4, cudaMemcpyDeviceToDevice, ctx->stream), "bias copy");
      } else {
        return set_err(ctx, PSV_EINVAL, "weight %d: device biases must be f32", i);
      }
    } else if (x.location == PSV_LOC_HOST) {
      std::vector<uint8_t> tmp;
      const void* src = x.data;
      size_t bytes = 0;
      if (matrix) {
        bytes = numel * 2;
        if (x.dtype == PSV_DTYPE_F32) {
          tmp.resize(bytes);
          const float* f = static_cast<const float*>(x.data);
          uint16_t* o = reinterpret_cast<uint16_t*>(tmp.data());
          for (int64_t k = 0; k < numel; ++k) o[k] = f32_to_bf16_bits(f[k]);
          src = tmp.data();
        }
      } else {
        bytes = numel * 4;
        if (x.dtype == PSV_DTYPE_BF16) {
          tmp.resize(bytes);
          const uint16_t* h = static_cast<const uint16_t*>(x.data);
          float* o = reinterpret_cast<float*>(tmp.data());
          for (int64_t k = 0; k < numel; ++k) o[k] = bf16_bits_to_f32(h[k]);
          src = tmp.data();
        }
      }
      CK(cudaMemcpyAsync(dst, src, bytes, cudaMemcpyHostToDevice, ctx->stream), "weight upload");
      CK(cudaStreamSynchronize(ctx->stream), "weight upload sync");
    } else {
      return set_err(ctx, PSV_EINVAL, "weight %d: bad location", i);
    }
    if (x.id == PSV_W_IN_W)
      CK(psv::launch_build_in2(reinterpret_cast<const __nv_bfloat16*>(ctx->arena + L.w_in),
                               reinterpret_cast<__nv_bfloat16*>(ctx->arena + L.w_in2), static_cast<int>(d),
                               static_cast<int>(C), L.K2, L.Npad_o, ctx->stream),
         "in-projection weight build");
    if (global) ctx->w_loaded[x.id] = true;
    else ctx->blk_loaded[static_cast<size_t>(x.block) * 16 + (x.id - PSV_W_QKV_W)] = 1;
  }
  if (!ctx->plan_only) CK(cudaStreamSynchronize(ctx->stream), "weight load sync");
  return PSV_OK;
}

static bool all_weights_loaded(const psv_ctx* ctx) {
  for (int id = PSV_W_IN_W; id <= PSV_W_OUT_B; ++id)
    if (!ctx->w_loaded[id]) return false;
  for (int b = 0; b < ctx->m.B; ++b)
    for (int k = 0; k < 10; ++k)
      if (!ctx->blk_loaded[static_cast<size_t>(b) * 16 + k]) return false;
  return true;
}

namespace {

// adaLN tables of conditioning table `tab` (a stream, or max_streams + a
// chunk slot) from the device vector cond [d]: for every step s,
// e_s = W_t2 SiLU(W_t1 emb(t_s) + b_t1) + b_t2 + cond,
// mod[tab][s] = W_mod SiLU(e_s) + b_mod (all blocks), fmod[tab][s] likewise.
cudaError_t build_cond_tables(psv_ctx* ctx, const float* cond, int tab) {
  const psv_model_desc& m = ctx->m;
  const Layout& L = ctx->L;
  const int S = m.S, E = m.t_embed, d = m.d;
  float* s_a1 = ctx->at<float>(L.scratch);
  float* s_e = s_a1 + static_cast<size_t>(8) * d;
  cudaStream_t st = ctx->stream;
  cudaError_t e;
  if ((e = psv::launch_cond_linear(ctx->at<float>(L.temb_in), S, E, ctx->at<__nv_bfloat16>(L.w_t1),
                                   ctx->at<float>(L.b_t1), nullptr, s_a1, d, 0, st)) != cudaSuccess)
    return e;
  if ((e = psv::launch_cond_linear(s_a1, S, d, ctx->at<__nv_bfloat16>(L.w_t2), ctx->at<float>(L.b_t2), cond, s_e,
                                   d, 1, st)) != cudaSuccess)
    return e;
  if ((e = psv::launch_cond_linear(s_e, S, d, ctx->at<__nv_bfloat16>(L.w_mod), ctx->at<float>(L.b_mod), nullptr,
                                   ctx->at<float>(L.mod) + static_cast<size_t>(tab) * S * m.B * 6 * d,
                                   m.B * 6 * d, 1, st)) != cudaSuccess)
    return e;
  return psv::launch_cond_linear(s_e, S, d, ctx->at<__nv_bfloat16>(L.w_fmod), ctx->at<float>(L.b_fmod), nullptr,
                                 ctx->at<float>(L.fmod) + static_cast<size_t>(tab) * S * 2 * d, 2 * d, 1, st);
}

}  // namespace

PSV_API int psv_open_stream(psv_ctx* ctx, const float* cond, int* stream_id) {
  if (int r = check_ctx(ctx)) return r;
  if (!stream_id || (!cond && !ctx->plan_only)) return set_err(ctx, PSV_EINVAL, "null argument");
  int sid = -1;
  for (int i = 0; i < static_cast<int>(ctx->streams.size()); ++i)
    if (!ctx->streams[i].open) { sid = i; break; }
  if (sid < 0) return set_err(ctx, PSV_EAGAIN, "all %d streams are open", ctx->m.max_streams);
  if (!ctx->plan_only) {
    if (!all_weights_loaded(ctx)) return set_err(ctx, PSV_EINVAL, "load every weight before opening a stream");
    const psv_model_desc& m = ctx->m;
    const Layout& L = ctx->L;
    const int d = m.d;
    cudaStream_t st = ctx->stream;
    std::memcpy(ctx->h_misc, cond, static_cast<size_t>(m.d) * 4);
    float* s_cond = ctx->at<float>(L.scratch) + static_cast<size_t>(8) * (m.t_embed + 2 * m.d);
    CK(cudaMemcpyAsync(s_cond, ctx->h_misc, static_cast<size_t>(m.d) * 4, cudaMemcpyHostToDevice, ctx->stream),
       "cond upload");
    CK(build_cond_tables(ctx, s_cond, sid), "adaLN tables");
    // Fresh rings: chunk 0 of the new stream must not see an old stream's keys
    // (it attends to slot 0 only, but masked tails must stay finite).
    const size_t ring_k = static_cast<size_t>(L.Lr) * d * 2, ring_v = static_cast<size_t>(d) * L.Lp * 2;
    const size_t per = static_cast<size_t>(m.B) * m.S;
    CK(cudaMemsetAsync(ctx->arena + L.k_ring + sid * per * ring_k, 0, per * ring_k, st), "ring clear");
    CK(cudaMemsetAsync(ctx->arena + L.vt_ring + sid * per * ring_v, 0, per * ring_v, st), "ring clear");
    CK(cudaStreamSynchronize(st), "open sync");
  }
  StreamState& s = ctx->streams[sid];
  s = StreamState();
  s.open = true;
  s.finish_wave.assign(ctx->inflight, -1);
  s.own_cond.assign(ctx->inflight, 0);
  *stream_id = sid;
  return PSV_OK;
}

namespace {
int submit_impl(psv_ctx* ctx, int sid, const float* noise, const float* cond, bool with_cond);
}  // namespace

PSV_API int psv_submit_chunk(psv_ctx* ctx, int sid, const float* noise) {
  return submit_impl(ctx, sid, noise, nullptr, false);
}

PSV_API int psv_submit_chunk_cond(psv_ctx* ctx, int sid, const float* noise, const float* cond) {
  if (int r = check_ctx(ctx)) return r;
  if (!(ctx->m.flags & PSV_FLAG_CHUNK_COND))
    return set_err(ctx, PSV_EINVAL, "per-chunk conditioning needs a context created with PSV_FLAG_CHUNK_COND");
  if (!cond && !ctx->plan_only) return set_err(ctx, PSV_EINVAL, "null cond");
  return submit_impl(ctx, sid, noise, cond, true);
}

namespace {
int submit_impl(psv_ctx* ctx, int sid, const float* noise, const float* cond, bool with_cond) {
  if (int r = check_ctx(ctx)) return r;
  if (sid < 0 || sid >= static_cast<int>(ctx->streams.size()) || !ctx->streams[sid].open)
    return set_err(ctx, PSV_EINVAL, "stream %d is not open", sid);
  StreamState& s = ctx->streams[sid];
  if (s.n_sub - s.n_polled >= ctx->inflight)
    return set_err(ctx, PSV_EAGAIN, "stream %d has %d chunks alive: poll first", sid, ctx->inflight);
  const int64_t c = s.n_sub;
  if (!ctx->plan_only) {
    if (!noise) return set_err(ctx, PSV_EINVAL, "null noise");
    const psv_model_desc& m = ctx->m;
    const int slot = sid * ctx->inflight + static_cast<int>(c % ctx->inflight);
    const size_t tc = static_cast<size_t>(m.T) * m.C;
    float* stage = ctx->h_noise + slot * tc;
    std::memcpy(stage, noise, tc * 4);
    CK(cudaMemcpyAsync(ctx->at<float>(ctx->L.state) + slot * tc, stage, tc * 4, cudaMemcpyHostToDevice, ctx->stream),
       "noise upload");
    // RoPE base angles of the chunk: (c*T) * theta^(-2j/dh), in f64.
    float2* rb = ctx->h_rope + static_cast<size_t>(slot) * (m.dh / 2);
    for (int j = 0; j < m.dh / 2; ++j) {
      const double ang = static_cast<double>(c) * m.T * std::pow(static_cast<double>(m.rope_theta), -2.0 * j / m.dh);
      rb[j] = make_float2(static_cast<float>(std::cos(ang)), static_cast<float>(std::sin(ang)));
    }
    CK(cudaMemcpyAsync(ctx->at<float2>(ctx->L.rope_base) + static_cast<size_t>(slot) * (m.dh / 2), rb,
                       static_cast<size_t>(m.dh / 2) * 8, cudaMemcpyHostToDevice, ctx->stream),
       "rope upload");
    if (with_cond) {
      // The slot's staging and table are free: its previous chunk was polled.
      float* hc = ctx->h_ccond + static_cast<size_t>(slot) * m.d;
      float* dc = ctx->at<float>(ctx->L.ccond) + static_cast<size_t>(slot) * m.d;
      std::memcpy(hc, cond, static_cast<size_t>(m.d) * 4);
      CK(cudaMemcpyAsync(dc, hc, static_cast<size_t>(m.d) * 4, cudaMemcpyHostToDevice, ctx->stream),
         "chunk cond upload");
      CK(build_cond_tables(ctx, dc, m.max_streams + slot), "chunk adaLN tables");
    }
  }
  s.own_cond[static_cast<size_t>(c % ctx->inflight)] = with_cond ? 1 : 0;
  s.n_sub += 1;
  return PSV_OK;
}
}  // namespace

PSV_API int psv_wave_plan(psv_ctx* ctx, psv_task* buf, int cap, int* n) {
  if (!ctx || !n || cap < 0 || (cap > 0 && !buf)) return PSV_EINVAL;
  std::vector<psv_task> tasks;
  plan_wave(ctx, &tasks);
  *n = static_cast<int>(tasks.size());
  for (int i = 0; i < std::min(cap, *n); ++i) buf[i] = tasks[i];
  return PSV_OK;
}

namespace {

// Fold every finished, timed steady wave into the per-task-count means.
void harvest_wave_times(psv_ctx* ctx) {
  for (WaveTiming& tm : ctx->wave_tm) {
    if (!tm.pending) continue;
    if (cudaEventQuery(tm.t1) != cudaSuccess) continue;
    tm.pending = false;
    float ms = 0.0f;
    if (!tm.full || cudaEventElapsedTime(&ms, tm.t0, tm.t1) != cudaSuccess) continue;
    WaveStat& w = ctx->wave_stats[tm.n_tasks];
    w.count += 1;
    w.mean_ms += (ms - w.mean_ms) / static_cast<double>(w.count);
  }
}

// Algorithmic FLOPs of a steady wave with n tasks (full windows): the block
// GEMMs, the window attention, the in-projection and the velocity head.
double steady_wave_flops(const psv_model_desc& m, int n) {
  const double T = m.T, d = m.d, F = m.F, C = m.C, B = m.B, Lk = static_cast<double>(m.W + 1) * m.T;
  const double per_task = 2.0 * T * B * (4.0 * d * d + 2.0 * d * F) + 4.0 * T * Lk * d * B + 4.0 * T * C * d;
  return per_task * n;
}

double predict_wave_ms(psv_ctx* ctx, int n_streams) {
  if (!ctx->plan_only) harvest_wave_times(ctx);
  const int n = n_streams * ctx->m.S;
  auto hit = ctx->wave_stats.find(n);
  if (hit != ctx->wave_stats.end() && hit->second.count > 0) return hit->second.mean_ms;
  int best = -1;
  for (const auto& kv : ctx->wave_stats)
    if (kv.second.count > 0 && (best < 0 || std::abs(kv.first - n) < std::abs(best - n))) best = kv.first;
  if (best > 0)
    return ctx->wave_stats[best].mean_ms * steady_wave_flops(ctx->m, n) / steady_wave_flops(ctx->m, best);
  constexpr double kUnmeasuredFlops = 1.0e15;  // 1 PFLOP/s until a wave was timed
  return steady_wave_flops(ctx->m, n) / kUnmeasuredFlops * 1e3;
}

}  // namespace

PSV_API int psv_predict_wave_ms(psv_ctx* ctx, int n_streams, double* ms) {
  if (int r = check_ctx(ctx)) return r;
  if (!ms || n_streams < 1 || n_streams > ctx->m.max_streams)
    return set_err(ctx, PSV_EINVAL, "need 1 <= n_streams <= %d", ctx->m.max_streams);
  *ms = predict_wave_ms(ctx, n_streams);
  return PSV_OK;
}

PSV_API int psv_admit_stream(psv_ctx* ctx, const float* cond, double slo_ms, int* stream_id,
                             double* predicted_ms) {
  if (int r = check_ctx(ctx)) return r;
  if (!stream_id) return set_err(ctx, PSV_EINVAL, "null stream_id");
  int n_open = 0;
  for (const StreamState& s : ctx->streams) n_open += s.open ? 1 : 0;
  if (n_open >= ctx->m.max_streams)
    return set_err(ctx, PSV_EAGAIN, "rejected: no KV ring set free (%d streams open)", n_open);
  const double pred = predict_wave_ms(ctx, n_open + 1);
  if (predicted_ms) *predicted_ms = pred;
  if (slo_ms > 0.0 && pred > slo_ms)
    return set_err(ctx, PSV_EAGAIN, "rejected: predicted %.3f ms per chunk > the stream's SLO %.3f ms", pred,
                   slo_ms);
  for (int i = 0; i < static_cast<int>(ctx->streams.size()); ++i) {
    const StreamState& s = ctx->streams[i];
    if (s.open && s.slo_ms > 0.0 && pred > s.slo_ms)
      return set_err(ctx, PSV_EAGAIN, "rejected: predicted %.3f ms per chunk > stream %d's SLO %.3f ms", pred, i,
                     s.slo_ms);
  }
  if (int r = psv_open_stream(ctx, cond, stream_id)) return r;
  ctx->streams[*stream_id].slo_ms = slo_ms > 0.0 ? slo_ms : 0.0;
  return PSV_OK;
}

PSV_API int psv_run_wave(psv_ctx* ctx, int* n_tasks) {
  if (int r = check_ctx(ctx)) return r;
  if (!n_tasks) return set_err(ctx, PSV_EINVAL, "null n_tasks");
  std::vector<psv_task> tasks;
  plan_wave(ctx, &tasks);
  const int n = static_cast<int>(tasks.size());
  *n_tasks = n;
  if (n == 0) return PSV_OK;
  if (!ctx->plan_only) {
    harvest_wave_times(ctx);
    WaveTiming& tm = ctx->wave_tm[ctx->wave_id % kWaveEvents];
    if (tm.pending) {
      // The slot's previous wave is 64 waves old; make sure it was counted.
      CK(cudaEventSynchronize(tm.t1), "wave timing");
      harvest_wave_times(ctx);
    }
    std::vector<TaskDev> dev(n);
    for (int i = 0; i < n; ++i) dev[i] = to_dev(ctx, tasks[i]);
    // Task table: pinned ring buffer, reused only after its copy finished.
    const int tb = ctx->task_buf;
    ctx->task_buf = (tb + 1) % kTaskBufs;
    CK(cudaEventSynchronize(ctx->task_ev[tb]), "task buffer reuse");
    TaskDev* h = ctx->h_tasks + static_cast<size_t>(tb) * ctx->L.max_tasks;
    std::memcpy(h, dev.data(), sizeof(TaskDev) * n);
    CK(cudaMemcpyAsync(ctx->at<TaskDev>(ctx->L.tasks), h, sizeof(TaskDev) * n, cudaMemcpyHostToDevice, ctx->stream),
       "task table upload");
    CK(cudaEventRecord(ctx->task_ev[tb], ctx->stream), "task event");
    tm.n_tasks = n;
    tm.full = true;
    for (const TaskDev& t : dev) tm.full = tm.full && t.kv_len == ctx->L.Lr;
    CK(cudaEventRecord(tm.t0, ctx->stream), "wave timing");
    const bool tap = ctx->tap_block >= 0;
    const bool eager = ctx->profiling || tap || !ctx->use_graphs;
    if (eager) {
      CK(enqueue_wave(ctx, ctx->stream, n, ctx->profiling, tap, &dev), "wave launch");
      ctx->tap_block = -1;
    } else {
      // A wave's launches depend on its task count and on how many attention
      // work pieces its windows make (fill waves have shorter windows).
      std::vector<int> kvl;
      for (const TaskDev& t : dev) kvl.push_back(t.kv_len);
      const int64_t key = (static_cast<int64_t>(n) << 32) |
                          static_cast<int64_t>(psv::attn_pieces(kvl.data(), n, ctx->m.T, ctx->m.H));
      int& seen = ctx->shape_seen[key];
      auto it = ctx->graphs.find(key);
      if (it == ctx->graphs.end() && seen >= 1) {
        // Captured on a private stream (capture is not allowed on the legacy
        // default stream a caller may pass); replayed on the caller's stream.
        cudaGraph_t g = nullptr;
        CK(cudaStreamBeginCapture(ctx->cap_stream, cudaStreamCaptureModeThreadLocal), "graph capture begin");
        cudaError_t le = enqueue_wave(ctx, ctx->cap_stream, n, false, false, &dev);
        cudaError_t ce = cudaStreamEndCapture(ctx->cap_stream, &g);
        if (le != cudaSuccess) return cuda_fail(ctx, le, "wave capture");
        if (ce != cudaSuccess) return cuda_fail(ctx, ce, "graph capture end");
        cudaGraphExec_t ex = nullptr;
        cudaError_t ie = cudaGraphInstantiate(&ex, g, 0);
        cudaGraphDestroy(g);
        if (ie != cudaSuccess) return cuda_fail(ctx, ie, "graph instantiate");
        it = ctx->graphs.emplace(key, ex).first;
      }
      if (it != ctx->graphs.end()) {
        CK(cudaGraphLaunch(it->second, ctx->stream), "graph launch");
      } else {
        CK(enqueue_wave(ctx, ctx->stream, n, false, false, &dev), "wave launch");
      }
      seen += 1;
    }
    CK(cudaEventRecord(ctx->wave_ev[ctx->wave_id % kWaveEvents], ctx->stream), "wave event");
    CK(cudaEventRecord(tm.t1, ctx->stream), "wave timing");
    // Profiled and tapped waves run eagerly with extra synchronisation: not
    // representative of the steady state.
    tm.pending = !eager;
  }
  for (const psv_task& t : tasks) {
    StreamState& s = ctx->streams[t.stream];
    s.done[t.step] += 1;
    if (t.step == ctx->m.S - 1) s.finish_wave[t.chunk % ctx->inflight] = ctx->wave_id;
  }
  ctx->wave_id += 1;
  return PSV_OK;
}

PSV_API int psv_poll_chunk(psv_ctx* ctx, int sid, float* out, int64_t* chunk_idx) {
  if (int r = check_ctx(ctx)) return r;
  if (sid < 0 || sid >= static_cast<int>(ctx->streams.size()) || !ctx->streams[sid].open)
    return set_err(ctx, PSV_EINVAL, "stream %d is not open", sid);
  StreamState& s = ctx->streams[sid];
  const int64_t c = s.n_polled;
  if (c >= s.done[ctx->m.S - 1]) return PSV_EAGAIN;
  if (!ctx->plan_only) {
    if (!out) return set_err(ctx, PSV_EINVAL, "null output buffer");
    const int64_t w = s.finish_wave[c % ctx->inflight];
    cudaError_t q = cudaEventQuery(ctx->wave_ev[w % kWaveEvents]);
    if (q == cudaErrorNotReady) return PSV_EAGAIN;
    if (q != cudaSuccess) return cuda_fail(ctx, q, "wave event query");
    if (int r = read_device_error(ctx)) return r;
    const psv_model_desc& m = ctx->m;
    const size_t tc = static_cast<size_t>(m.T) * m.C;
    const int slot = sid * ctx->inflight + static_cast<int>(c % ctx->inflight);
    CK(cudaMemcpyAsync(ctx->h_out, ctx->at<float>(ctx->L.state) + slot * tc, tc * 4, cudaMemcpyDeviceToHost,
                       ctx->copy_stream), "output copy");
    CK(cudaStreamSynchronize(ctx->copy_stream), "output copy sync");
    std::memcpy(out, ctx->h_out, tc * 4);
  }
  if (chunk_idx) *chunk_idx = c;
  s.n_polled += 1;
  return PSV_OK;
}

PSV_API int psv_sync(psv_ctx* ctx, int timeout_ms) {
  if (int r = check_ctx(ctx)) return r;
  if (ctx->plan_only) return PSV_OK;
  const auto t0 = std::chrono::steady_clock::now();
  for (;;) {
    cudaError_t q = cudaStreamQuery(ctx->stream);
    if (q == cudaSuccess) break;
    if (q != cudaErrorNotReady) return cuda_fail(ctx, q, "stream query");
    if (timeout_ms >= 0) {
      const auto ms = std::chrono::duration_cast<std::chrono::milliseconds>(std::chrono::steady_clock::now() - t0).count();
      if (ms >= timeout_ms) return set_err(ctx, PSV_ETIMEDOUT, "psv_sync: %d ms passed", timeout_ms);
    }
    std::this_thread::sleep_for(std::chrono::microseconds(50));
  }
  return read_device_error(ctx);
}

PSV_API int psv_close_stream(psv_ctx* ctx, int sid) {
  if (!ctx) return PSV_EINVAL;
  if (sid < 0 || sid >= static_cast<int>(ctx->streams.size()) || !ctx->streams[sid].open)
    return set_err(ctx, PSV_EINVAL, "stream %d is not open", sid);
  ctx->streams[sid].open = false;
  return PSV_OK;
}

PSV_API void psv_destroy(psv_ctx* ctx) {
  if (!ctx) return;
  if (!ctx->plan_only) {
    if (ctx->stream || ctx->arena) cudaStreamSynchronize(ctx->stream);
    for (auto& kv : ctx->graphs) cudaGraphExecDestroy(kv.second);
    for (auto& r : ctx->prof) {
      cudaEventDestroy(r.a);
      cudaEventDestroy(r.b);
    }
    for (cudaEvent_t e : ctx->ev_pool) cudaEventDestroy(e);
    for (int i = 0; i < kTaskBufs; ++i)
      if (ctx->task_ev[i]) cudaEventDestroy(ctx->task_ev[i]);
    for (int i = 0; i < kWaveEvents; ++i)
      if (ctx->wave_ev[i]) cudaEventDestroy(ctx->wave_ev[i]);
    for (int i = 0; i < kWaveEvents; ++i) {
      if (ctx->wave_tm[i].t0) cudaEventDestroy(ctx->wave_tm[i].t0);
      if (ctx->wave_tm[i].t1) cudaEventDestroy(ctx->wave_tm[i].t1);
    }
    if (ctx->h_tasks) cudaFreeHost(ctx->h_tasks);
    if (ctx->h_noise) cudaFreeHost(ctx->h_noise);
    if (ctx->h_rope) cudaFreeHost(ctx->h_rope);
    if (ctx->h_out) cudaFreeHost(ctx->h_out);
    if (ctx->h_misc) cudaFreeHost(ctx->h_misc);
    if (ctx->h_ccond) cudaFreeHost(ctx->h_ccond);
    if (ctx->copy_stream) cudaStreamDestroy(ctx->copy_stream);
    if (ctx->cap_stream) cudaStreamDestroy(ctx->cap_stream);
  }
  delete ctx;
}

PSV_API const char* psv_last_error(const psv_ctx* ctx) {
  return ctx ? ctx->err.c_str() : g_create_error.c_str();
}

PSV_API int psv_set_graphs(psv_ctx* ctx, int enabled) {
  if (!ctx) return PSV_EINVAL;
  ctx->use_graphs = enabled != 0;
  return PSV_OK;
}

PSV_API int psv_set_profiling(psv_ctx* ctx, int enabled) {
  if (int r = check_ctx(ctx)) return r;
  if (enabled && !ctx->profiling) {
    for (int k = 0; k < K_COUNT; ++k) {
      ctx->kind_ms[k] = ctx->kind_flops[k] = ctx->kind_bytes[k] = 0.0;
      ctx->kind_launches[k] = 0;
    }
  }
  if (!enabled && ctx->profiling && !ctx->plan_only) {
    if (int r = collect_profile(ctx)) return r;
  }
  ctx->profiling = enabled != 0;
  return PSV_OK;
}

PSV_API int psv_kernel_times(psv_ctx* ctx, psv_kernel_time* out, int cap, int* n) {
  if (int r = check_ctx(ctx)) return r;
  if (!n || cap < 0 || (cap > 0 && !out)) return set_err(ctx, PSV_EINVAL, "bad arguments");
  if (!ctx->plan_only)
    if (int r = collect_profile(ctx)) return r;
  *n = K_COUNT;
  for (int k = 0; k < std::min(cap, static_cast<int>(K_COUNT)); ++k) {
    std::memset(&out[k], 0, sizeof(psv_kernel_time));
    std::snprintf(out[k].name, sizeof(out[k].name), "%s", kKindNames[k]);
    out[k].launches = ctx->kind_launches[k];
    out[k].total_ms = ctx->kind_ms[k];
    out[k].flops = ctx->kind_flops[k];
    out[k].bytes = ctx->kind_bytes[k];
  }
  return PSV_OK;
}

PSV_API int psv_debug_tap(psv_ctx* ctx, int block, float* h_in, float* h_out) {
  if (int r = check_ctx(ctx)) return r;
  if (block < 0 || block >= ctx->m.B || !h_in || !h_out) return set_err(ctx, PSV_EINVAL, "bad tap arguments");
  ctx->tap_block = block;
  ctx->tap_in = h_in;
  ctx->tap_out = h_out;
  return PSV_OK;
}

PSV_API int psv_debug_error_word(psv_ctx* ctx, size_t* arena_offset) {
  if (!ctx || !arena_offset) return PSV_EINVAL;
  if (ctx->plan_only) return set_err(ctx, PSV_EINVAL, "plan-only context has no error word");
  *arena_offset = ctx->L.err;
  return PSV_OK;
}

PSV_API int psv_debug_read_kv(psv_ctx* ctx, int sid, int block, int step, float* k, float* v) {
  if (int r = check_ctx(ctx)) return r;
  const psv_model_desc& m = ctx->m;
  if (ctx->plan_only || sid < 0 || sid >= m.max_streams || block < 0 || block >= m.B || step < 0 || step >= m.S ||
      !k || !v)
    return set_err(ctx, PSV_EINVAL, "bad kv read arguments");
  const Layout& L = ctx->L;
  const int ring = (sid * m.B + block) * m.S + step;
  const size_t nk = static_cast<size_t>(L.Lr) * m.d, nv = static_cast<size_t>(m.d) * L.Lp;
  std::vector<uint16_t> hk(nk), hv(nv);
  CK(cudaStreamSynchronize(ctx->stream), "kv read sync");
  CK(cudaMemcpy(hk.data(), ctx->arena + L.k_ring + ring * nk * 2, nk * 2, cudaMemcpyDeviceToHost), "kv read");
  CK(cudaMemcpy(hv.data(), ctx->arena + L.vt_ring + ring * nv * 2, nv * 2, cudaMemcpyDeviceToHost), "kv read");
  for (size_t i = 0; i < nk; ++i) k[i] = bf16_bits_to_f32(hk[i]);
  for (int r = 0; r < L.Lr; ++r)
    for (int c = 0; c < m.d; ++c) {
      const int head = c / m.dh, e = c % m.dh;
      v[static_cast<size_t>(r) * m.d + c] = bf16_bits_to_f32(hv[(static_cast<size_t>(head) * m.dh + e) * L.Lp + r]);
    }
  return PSV_OK;
}
