// Persistent tcgen05 GEMM with fused epilogues:  C = A W^T + bias.
//
// A [M, K] bf16 activations and W [N, K] bf16 weights (nn.Linear layout)
// are both K-major, so TMA loads 128-byte-swizzled tiles that feed
// tcgen05.mma directly.  CTAs run in pairs (a cluster of two SMs) on 256x256
// output tiles (256x512 for the long-K down-projection, see GemmShape) with
// 2-SM MMAs (cta_group::2, M = 256): each CTA stages its own 128 rows of A and
// one 128-row half of the W tile (64 KB per 128-wide k-block, 3 stages), and
// the even CTA issues every MMA for both.  Per SM this halves the weight
// traffic and leaves room for a deep TMA pipeline.  Warp roles:
//   warp 0      TMA producer (both CTAs; completion signalled on the even
//               CTA's stage barrier)
//   warp 1      TMEM allocator (both CTAs) + MMA issuer (even CTA only):
//               256x256x16 MMAs into a double-buffered 2 x 256-column TMEM
//               accumulator (one 512-column accumulator for the wide tile)
//   warps 2..9  epilogue: tcgen05.ld of this CTA's 128 rows, two warps per
//               TMEM lane quadrant (128 columns each), the fused epilogue.
// The tile shape and the K order are fixed for every M, so a row's result
// does not depend on which other tasks share the wave (batch invariance).
//
// The epilogues implement the block's linear layers (gated residual adds,
// GELU MLP, QKV with RoPE and the noisy-KV append of the pages: a chunk's
// keys/values at (block, step) stay resident for its W successors; AREX
// article "vLLM 与 Physis-AI 联合介绍 PhysisServe 推理系统", §难题).
#include "psv_device.cuh"
#include "psv_kernels.h"

namespace psv {

namespace {

constexpr int BM = kGemmBM;
constexpr uint32_t TMEM_COLS = 512;
constexpr int EPI_WARPS = 8;
constexpr int STAGE_BYTES = 32 * 32 * 4;    // per epilogue warp: a 32 x 32 f32 box
constexpr uint32_t IDESC = umma_idesc_bf16(2 * BM, 256);  // 256 x 256 per 2-SM MMA

// Pair tile shapes.  Narrow: 256 x 256 per pair, 128-wide k-blocks in 3
// stages, a double-buffered 2 x 256-column TMEM accumulator (the epilogue of
// one tile overlaps the MMAs of the next).  Wide: 256 x 512 per pair (two
// N = 256 MMAs per k-step into all 512 TMEM columns), 64-wide k-blocks in 4
// stages: a quarter fewer operand bytes per FLOP — the main loop is bound by
// how fast TMA fills one SM's shared memory — at the price of a single
// accumulator, so the epilogue is no longer hidden.
template <bool WIDE>
struct GemmShape {
  static constexpr int BN = WIDE ? 512 : 256;   // pair tile width
  static constexpr int BK = WIDE ? 64 : 128;
  static constexpr int STAGES = WIDE ? 4 : 3;
  static constexpr int NSLAB = BN / 256;        // N = 256 MMAs per k-step
  static constexpr int KA = BK / 64;            // 128-byte swizzle atoms along K per stage
  static constexpr int A_ATOM = BM * 128;       // 16 KB: 128 rows x 64 k
  static constexpr int B_ATOM = 128 * 128;      // 16 KB: 128 W rows x 64 k
  static constexpr int A_BYTES = KA * A_ATOM;   // this CTA's 128 rows of A
  static constexpr int B_SLAB = KA * B_ATOM;    // this CTA's 128-row half of one N = 256 slab
  static constexpr int B_BYTES = NSLAB * B_SLAB;
  static constexpr int ACC_BUFS = WIDE ? 1 : 2;
  static constexpr size_t SMEM =
      1024 + STAGES * (A_BYTES + B_BYTES) + EPI_WARPS * STAGE_BYTES + (2 * STAGES + 4) * 8 + 16;
  static_assert(SMEM <= 232448, "GEMM shared memory over the per-block limit");
};

// tanh.approx.f32: the SFU's tanh (max relative error ~2^-11, far below the
// bf16 rounding of the GELU output).
__device__ __forceinline__ float tanh_approx(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float gelu_tanh(float x) {
  const float k0 = 0.7978845608028654f;  // sqrt(2/pi)
  const float x2 = x * x;
  return 0.5f * x * (1.0f + tanh_approx(k0 * x * fmaf(0.044715f, x2, 1.0f)));
}

// RoPE of 32 consecutive q or k columns of one row, starting at element e0 of
// a head: rotate pairs (e, e+1) by angle (c*T + li) * f_{e/2}; the angle is
// assembled from two tables built in f64 on the host.
__device__ __forceinline__ void qk_rope32(const GemmParams& p, const TaskDev& t, int li, int e0,
                                          float* v) {
  const float2* rb = p.rope_base + static_cast<int64_t>(t.rope_slot) * (p.dh >> 1) + (e0 >> 1);
  // in-chunk table is [dh/2][T]: the warp's 32 rows read 32 consecutive entries
  const float2* rl = p.rope_local + static_cast<int64_t>(e0 >> 1) * p.T + li;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const float2 cb = __ldg(rb + i);
    const float2 cl = __ldg(rl + static_cast<int64_t>(i) * p.T);
    const float cs = cb.x * cl.x - cb.y * cl.y;
    const float sn = cb.y * cl.x + cb.x * cl.y;
    const float a = v[2 * i], b = v[2 * i + 1];
    v[2 * i] = a * cs - b * sn;
    v[2 * i + 1] = a * sn + b * cs;
  }
}

// Fused epilogue of 32 consecutive columns [n0, n0+32) of one row, written
// row by row (velocity head; V^T and the q/k rows that qkv_chunk64 cannot
// write as one box).
template <int EPI>
__device__ __forceinline__ void epilogue32(const GemmParams& p, int row, int n0, float* v) {
  if (row >= p.M || n0 >= p.N) return;
  const int ti = row / p.T;
  const TaskDev& t = p.tasks[ti];
  const int li = row - t.row0;  // token index within the chunk

  if (EPI == EPI_EULER) {
    // Velocity head: x += dt * (acc + b_out); only the first C columns exist.
    // Every load of x and b_out is issued before the first store (one
    // dependent read-modify-write per element would serialise 32 round trips
    // to memory per row); 16-byte accesses where the row allows them.
    float* x = p.state + (static_cast<int64_t>(t.state_slot) * p.T + li) * p.C + n0;
    const float* bn = p.bias + n0;
    const int nn = p.N - n0 < 32 ? p.N - n0 : 32;
    if (nn == 32 && (p.C % 4) == 0) {
      float4 xv[8], bv[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        xv[i] = *reinterpret_cast<const float4*>(x + 4 * i);
        bv[i] = __ldg(reinterpret_cast<const float4*>(bn) + i);
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        float4 r;
        r.x = xv[i].x + t.dt * (v[4 * i] + bv[i].x);
        r.y = xv[i].y + t.dt * (v[4 * i + 1] + bv[i].y);
        r.z = xv[i].z + t.dt * (v[4 * i + 2] + bv[i].z);
        r.w = xv[i].w + t.dt * (v[4 * i + 3] + bv[i].w);
        *reinterpret_cast<float4*>(x + 4 * i) = r;
      }
    } else {
      float xv[32], bv[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        xv[i] = i < nn ? x[i] : 0.0f;
        bv[i] = i < nn ? __ldg(bn + i) : 0.0f;
      }
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (i < nn) x[i] = xv[i] + t.dt * (v[i] + bv[i]);
    }
    return;
  }

  const float4* b4 = reinterpret_cast<const float4*>(p.bias + n0);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float4 bb = __ldg(b4 + i);
    v[4 * i] += bb.x;
    v[4 * i + 1] += bb.y;
    v[4 * i + 2] += bb.z;
    v[4 * i + 3] += bb.w;
  }

  if (EPI == EPI_QKV) {
    const int sec = n0 / p.d;  // 0 = q, 1 = k, 2 = v
    const int j0 = n0 - sec * p.d;
    const int head = j0 / p.dh;
    const int e0 = j0 - head * p.dh;
    if (sec < 2) qk_rope32(p, t, li, e0, v);
    const int ring = t.ring0 + p.block * p.S;
    const int rr = t.slot * p.T + li;  // row inside the ring
    if (sec == 2) {
      // V is stored transposed per head ([dh][Lp]) so that the P.V MMA reads
      // it K-major; lanes hold consecutive tokens, so each store of the warp
      // covers 32 consecutive keys.
      __nv_bfloat16* vt = p.vt_ring +
                          ((static_cast<int64_t>(ring) * p.H + head) * p.dh + e0) * p.Lp + rr;
#pragma unroll
      for (int i = 0; i < 32; ++i) vt[static_cast<int64_t>(i) * p.Lp] = __float2bfloat16_rn(v[i]);
    } else {
      __nv_bfloat16* dst =
          (sec == 0) ? p.q_out + static_cast<int64_t>(row) * p.d + j0
                     : p.k_ring + (static_cast<int64_t>(ring) * p.Lr + rr) * p.d + j0;
      uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        uint4 w;
        w.x = pack_bf16x2(v[8 * i + 0], v[8 * i + 1]);
        w.y = pack_bf16x2(v[8 * i + 2], v[8 * i + 3]);
        w.z = pack_bf16x2(v[8 * i + 4], v[8 * i + 5]);
        w.w = pack_bf16x2(v[8 * i + 6], v[8 * i + 7]);
        d4[i] = w;
      }
    }
  }
}

// ---- gated residual through a TMA reduce-add: h[rows][cols] += box.
__device__ __forceinline__ void tma_reduce_add_2d(const CUtensorMap* map, const void* src, int x,
                                                  int y) {
  asm volatile(
      "cp.reduce.async.bulk.tensor.2d.global.shared::cta.add.tile.bulk_group [%0, {%2, %3}], [%1];"
      ::"l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(src)), "r"(x), "r"(y)
      : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Until the source shared memory of every committed bulk operation was read.
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Gated residual of one warp's 32 rows x 32 columns: h += gate * (acc + b).
// The products are staged as a 128-byte-swizzled [32][32] f32 box and added
// into h by one TMA reduce (the add happens in L2 on whole lines, instead of
// 32 partial-line read-modify-writes per warp instruction).  Every element
// gets exactly one add, so the result is deterministic.  Rows past M add 0.
__device__ __forceinline__ void resid_chunk(const GemmParams& p, const CUtensorMap* tmC,
                                            float* stage, int row, int row0, int n0, float* v) {
  const int lane = lane_id();
  if (row < p.M && n0 < p.N) {
    const TaskDev& t = p.tasks[row / p.T];
    const float4* b4 = reinterpret_cast<const float4*>(p.bias + n0);
    const float4* g4 = reinterpret_cast<const float4*>(
        p.mod + t.mod0 + static_cast<int64_t>(p.block) * 6 * p.d + p.gate_off + n0);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float4 bb = __ldg(b4 + i), g = __ldg(g4 + i);
      v[4 * i] = g.x * (v[4 * i] + bb.x);
      v[4 * i + 1] = g.y * (v[4 * i + 1] + bb.y);
      v[4 * i + 2] = g.z * (v[4 * i + 2] + bb.z);
      v[4 * i + 3] = g.w * (v[4 * i + 3] + bb.w);
    }
  } else {
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = 0.0f;
  }
  // The previous box of this warp must have been read out of the staging buffer.
  if (lane == 0) bulk_wait_read();
  __syncwarp();
  float4* st4 = reinterpret_cast<float4*>(stage);
#pragma unroll
  for (int j = 0; j < 8; ++j)
    st4[lane * 8 + (j ^ (lane & 7))] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) {
    tma_reduce_add_2d(tmC, stage, n0, row0);
    bulk_commit();
  }
}

__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, const void* src, int x, int y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%2, %3}], [%1];"
               ::"l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(src)), "r"(x), "r"(y)
               : "memory");
}

// Plain f32 output of one warp's 32 rows x 32 columns: h = acc + b, staged as
// a 128-byte-swizzled [32][32] f32 box and written by one TMA store (the
// in-projection, which writes the residual stream of the wave's rows).
__device__ __forceinline__ void store_chunk(const GemmParams& p, const CUtensorMap* tmC,
                                            float* stage, int row0, int n0, float* v) {
  const int lane = lane_id();
  if (n0 >= p.N) return;
  const float4* b4 = reinterpret_cast<const float4*>(p.bias + n0);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float4 bb = __ldg(b4 + i);
    v[4 * i] += bb.x;
    v[4 * i + 1] += bb.y;
    v[4 * i + 2] += bb.z;
    v[4 * i + 3] += bb.w;
  }
  if (lane == 0) bulk_wait_read();
  __syncwarp();
  float4* st4 = reinterpret_cast<float4*>(stage);
#pragma unroll
  for (int j = 0; j < 8; ++j)
    st4[lane * 8 + (j ^ (lane & 7))] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) {
    tma_store_2d(tmC, stage, n0, row0);
    bulk_commit();
  }
}

// GELU of one warp's 32 rows x 64 columns, staged as a 128-byte-swizzled
// [32][64] bf16 box and written by one TMA store (whole 128-byte lines).
// Rows past M are written as zeros.
__device__ __forceinline__ void gelu_chunk64(const GemmParams& p, const CUtensorMap* tmC,
                                             void* stage, int row, int row0, int n0, float* v) {
  const int lane = lane_id();
  uint32_t w[32];
  if (row < p.M) {
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const int n = n0 + 2 * i;
      const float b0 = n < p.N ? __ldg(p.bias + n) : 0.0f;
      const float b1 = n + 1 < p.N ? __ldg(p.bias + n + 1) : 0.0f;
      w[i] = pack_bf16x2(gelu_tanh(v[2 * i] + b0), gelu_tanh(v[2 * i + 1] + b1));
    }
  } else {
#pragma unroll
    for (int i = 0; i < 32; ++i) w[i] = 0u;
  }
  if (lane == 0) bulk_wait_read();
  __syncwarp();
  uint4* st4 = reinterpret_cast<uint4*>(stage);
#pragma unroll
  for (int j = 0; j < 8; ++j)
    st4[lane * 8 + (j ^ (lane & 7))] = make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) {
    tma_store_2d(tmC, stage, n0, row0);
    bulk_commit();
  }
}

__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, const void* src, int x, int y,
                                             int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4}], [%1];"
      ::"l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(src)), "r"(x), "r"(y), "r"(z)
      : "memory");
}

// V^T of one warp's 32 rows x 64 columns [n0, n0 + 64) of the v section:
// per 32 columns (one head, dims e0..e0+31) a [32 dims][32 tokens] bf16 box,
// transposed through the warp's staging buffer and written by one TMA store
// into the task's ring rows of the transposed V ring (tme: [rings*H][dh][Lp],
// 32 x 32 boxes, no swizzle).  The caller checks that the warp's rows lie in
// one task and below M, and that ring rows start 8-aligned (T % 8 == 0).
__device__ __forceinline__ void vt_chunk64(const GemmParams& p, const CUtensorMap* tme, void* stage,
                                           int row0, int n0, float* v) {
  const int lane = lane_id();
  const TaskDev& t = p.tasks[row0 / p.T];
  const int rr0 = t.slot * p.T + (row0 - t.row0);  // first ring row of the warp's tokens
  const int ring = t.ring0 + p.block * p.S;
  uint16_t* st16 = reinterpret_cast<uint16_t*>(stage);
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int j = n0 + 32 * h - 2 * p.d;
    const int head = j / p.dh, e0 = j - head * p.dh;
    const float4* b4 = reinterpret_cast<const float4*>(p.bias + n0 + 32 * h);
    float* vh = v + 32 * h;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float4 bb = __ldg(b4 + i);
      vh[4 * i] += bb.x;
      vh[4 * i + 1] += bb.y;
      vh[4 * i + 2] += bb.z;
      vh[4 * i + 3] += bb.w;
    }
    if (lane == 0) bulk_wait_read();
    __syncwarp();
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const __nv_bfloat16 b = __float2bfloat16_rn(vh[i]);
      st16[i * 32 + lane] = *reinterpret_cast<const uint16_t*>(&b);
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      tma_store_3d(tme, stage, rr0, e0, ring * p.H + head);
      bulk_commit();
    }
  }
}

// QKV epilogue of one warp's 32 rows x 64 columns [n0, n0 + 64).  q and k
// (bias, RoPE) are staged as a 128-byte-swizzled [32][64] bf16 box and
// written by one TMA store: q into [rows][d] (tmq), k into the task's ring
// rows (tmk: [rings][Lr][d]) — whole 128-byte lines instead of 32 partial
// lines per warp store.  The box needs all 32 rows in one task and below M
// (a box must not reach into the next task's ring rows); the few warps that
// straddle a task boundary, and V^T (stored transposed), go row by row.
__device__ __forceinline__ void qkv_chunk64(const GemmParams& p, const CUtensorMap* tmq,
                                            const CUtensorMap* tmk, const CUtensorMap* tmv,
                                            void* stage, int row, int row0, int n0, float* v) {
  if (n0 >= p.N) return;
  const int sec = n0 / p.d;
  const int last = row0 + 31;
  if (sec == 2 && p.vt_box && (p.dh % 32) == 0 && last < p.M && row0 / p.T == last / p.T) {
    vt_chunk64(p, tmv, stage, row0, n0, v);
    return;
  }
  const bool box = (p.d % 64) == 0 && sec < 2 && last < p.M && row0 / p.T == last / p.T;
  if (!box) {
    epilogue32<EPI_QKV>(p, row, n0, v);
    epilogue32<EPI_QKV>(p, row, n0 + 32, v + 32);
    return;
  }
  const int lane = lane_id();
  const TaskDev& t = p.tasks[row / p.T];
  const int li = row - t.row0;
  const int j0 = n0 - sec * p.d;
  uint32_t w[32];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    float* vh = v + 32 * h;
    const float4* b4 = reinterpret_cast<const float4*>(p.bias + n0 + 32 * h);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float4 bb = __ldg(b4 + i);
      vh[4 * i] += bb.x;
      vh[4 * i + 1] += bb.y;
      vh[4 * i + 2] += bb.z;
      vh[4 * i + 3] += bb.w;
    }
    const int jh = j0 + 32 * h;
    qk_rope32(p, t, li, jh - (jh / p.dh) * p.dh, vh);
  }
#pragma unroll
  for (int i = 0; i < 32; ++i) w[i] = pack_bf16x2(v[2 * i], v[2 * i + 1]);
  if (lane == 0) bulk_wait_read();
  __syncwarp();
  uint4* st4 = reinterpret_cast<uint4*>(stage);
#pragma unroll
  for (int j = 0; j < 8; ++j)
    st4[lane * 8 + (j ^ (lane & 7))] = make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) {
    if (sec == 0) {
      tma_store_2d(tmq, stage, j0, row0);
    } else {
      const TaskDev& t0 = p.tasks[row0 / p.T];
      tma_store_3d(tmk, stage, j0, t0.slot * p.T + (row0 - t0.row0), t0.ring0 + p.block * p.S);
    }
    bulk_commit();
  }
}

// Warp-uniform bounded wait: lane 0 polls, the verdict is broadcast.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, int* err, int code) {
  int ok = 0;
  if (lane_id() == 0) ok = mbar_wait(bar, parity, err, code) ? 1 : 0;
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

template <int EPI, bool WIDE>
__global__ void __launch_bounds__(320, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA,
                   const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmC,
                   const __grid_constant__ CUtensorMap tmD,
                   const __grid_constant__ CUtensorMap tmE, const GemmParams p) {
  using G = GemmShape<WIDE>;
  constexpr int BN = G::BN, BK = G::BK, STAGES = G::STAGES, KA = G::KA;
  constexpr int A_ATOM = G::A_ATOM, B_ATOM = G::B_ATOM, A_BYTES = G::A_BYTES, B_BYTES = G::B_BYTES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * A_BYTES;
  uint8_t* sC = sB + STAGES * B_BYTES;  // epilogue staging, STAGE_BYTES per epilogue warp
  uint64_t* full = reinterpret_cast<uint64_t*>(sC + EPI_WARPS * STAGE_BYTES);  // even CTA
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + 2;                                         // used in the even CTA
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tempty + 2);

  pdl_trigger();
  const int warp = warp_id(), lane = lane_id();
  const int n_m = (p.M + BM - 1) / BM;
  const int n_n = (p.N + BN - 1) / BN;
  const int nk = (p.K + BK - 1) / BK;
  // Tile pairs (m-blocks 2i, 2i+1; same n-block), one per CTA pair at a time,
  // n-blocks fastest: the pairs running together share their activation
  // tiles (read from HBM once), and every weight tile stays L2-resident.
  const int rank = static_cast<int>(cluster_ctarank());
  const bool leader = rank == 0;
  const int cid = blockIdx.x >> 1, n_clusters = gridDim.x >> 1;
  const int n_mp = (n_m + 1) >> 1;
  const int n_pt = n_mp * n_n;

  if (warp == 0 && lane == 0) {
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(&full[i], 1);   // the even CTA's producer arrives (with all 64 KB of tx)
      mbar_init(&empty[i], 1);  // the 2-SM MMA commit arrives in both CTAs
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tfull[i], 1);
      mbar_init(&tempty[i], 16);  // 8 epilogue warps of each CTA
    }
    fence_mbar_init();
    prefetch_tensormap(&tmA);
    prefetch_tensormap(&tmB);
  }
  if (warp == 1) tmem_alloc_pair(tmem_slot, TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // The peer's barriers must be initialised before anything signals them.
  cluster_sync();
  const uint32_t tmem = *tmem_slot;
  // Everything above overlaps the previous kernel's tail; from here on the
  // kernel reads what it wrote.
  pdl_wait();

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer (both CTAs)
      const uint32_t full0 = mapa_shared(&full[0], 0);  // the even CTA's stage barriers
      int it = 0;
      bool ok = true;
      for (int tp = cid; tp < n_pt && ok; tp += n_clusters) {
        const int mb = 2 * (tp / n_n) + rank, nb = tp % n_n;
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int st = it % STAGES;
          const uint32_t ph = (it / STAGES) & 1;
          if (!mbar_wait(&empty[st], ph ^ 1, p.err, ERR_GEMM_TIMEOUT)) {
            ok = false;
            break;
          }
          if (leader) mbar_arrive_expect_tx(&full[st], 2 * (A_BYTES + B_BYTES));
          const uint32_t bar = full0 + st * 8;
#pragma unroll
          for (int a = 0; a < KA; ++a) {
            tma_load_2d_pair(sA + st * A_BYTES + a * A_ATOM, &tmA, bar, kb * BK + a * 64, mb * BM);
#pragma unroll
            for (int sl = 0; sl < G::NSLAB; ++sl)
              tma_load_3d_pair(sB + st * B_BYTES + sl * G::B_SLAB + a * B_ATOM, &tmB, bar,
                               kb * BK + a * 64, nb * BN + sl * 256 + rank * 128, p.wz);
          }
        }
      }
      // Wait until the MMAs released the last stages: nothing may still read
      // this CTA's shared memory or signal it after it leaves (bounded).
      const uint64_t t0 = global_timer_ns();
      for (int j = (it > STAGES ? it - STAGES : 0); j < it; ++j) {
        while (!mbar_try_wait(&empty[j % STAGES], (j / STAGES) & 1)) {
          if (global_timer_ns() - t0 > kWaitLimitNs) break;
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // ---------------- MMA issuer (even CTA), 2-SM MMAs for the pair
      int it = 0, tc = 0;
      bool ok = true;
      const uint64_t a_desc0 = umma_desc_kmajor(smem_u32(sA), 128);
      const uint64_t b_desc0 = umma_desc_kmajor(smem_u32(sB), 128);
      for (int tp = cid; tp < n_pt && ok; tp += n_clusters, ++tc) {
        const int acc = tc % G::ACC_BUFS;
        const uint32_t aph = (tc / G::ACC_BUFS) & 1;
        if (!mbar_wait(&tempty[acc], aph ^ 1, p.err, ERR_GEMM_TIMEOUT)) break;
        tc_fence_after();
        const uint32_t dtm = tmem + acc * 256;
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int st = it % STAGES;
          const uint32_t ph = (it / STAGES) & 1;
          if (!mbar_wait(&full[st], ph, p.err, ERR_GEMM_TIMEOUT)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t a = a_desc0 + static_cast<uint64_t>((st * A_BYTES) >> 4);
          const uint64_t b = b_desc0 + static_cast<uint64_t>((st * B_BYTES) >> 4);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k) {
            // k-step k: atom k / 4, 32 bytes per step inside the atom
            const uint32_t oa = ((k >> 2) * A_ATOM + (k & 3) * 32) >> 4;
            const uint32_t ob = ((k >> 2) * B_ATOM + (k & 3) * 32) >> 4;
#pragma unroll
            for (int sl = 0; sl < G::NSLAB; ++sl)
              umma_bf16_pair(dtm + sl * 256, a + oa, b + ((sl * G::B_SLAB) >> 4) + ob, IDESC,
                             (kb | k) != 0);
          }
          umma_commit_pair_mc(&empty[st], 0x3);  // free stage st in both CTAs
        }
        if (ok) umma_commit_pair_mc(&tfull[acc], 0x3);
      }
    }
  } else {
    // ---------------- epilogue warps (TMEM lane quadrant = warp % 4)
    const int q = warp & 3;
    const int chalf = (warp - 2) >> 2;  // which 128 accumulator columns
    const uint32_t tempty0 = mapa_shared(&tempty[0], 0);
    float* stage = reinterpret_cast<float*>(sC + (warp - 2) * STAGE_BYTES);
    int tc = 0;
    for (int tp = cid; tp < n_pt; tp += n_clusters, ++tc) {
      const int mb = 2 * (tp / n_n) + rank, nb = tp % n_n;
      const int acc = tc % G::ACC_BUFS;
      const uint32_t aph = (tc / G::ACC_BUFS) & 1;
      if (!warp_wait(&tfull[acc], aph, p.err, ERR_GEMM_TIMEOUT)) break;
      tc_fence_after();
      const int row = mb * BM + q * 32 + lane;
      const uint32_t tbase = tmem + acc * 256 + (static_cast<uint32_t>(q * 32) << 16);
      if constexpr (EPI == EPI_GELU || EPI == EPI_QKV) {
#pragma unroll 1
        for (int ch = chalf * (BN / 64); ch < (chalf + 1) * (BN / 64); ch += 2) {
          float v[64];
          tmem_ld32(tbase + ch * 32, v);
          tmem_ld32(tbase + ch * 32 + 32, v + 32);
          tmem_wait_ld();
          if constexpr (EPI == EPI_GELU)
            gelu_chunk64(p, &tmC, stage, row, mb * BM + q * 32, nb * BN + ch * 32, v);
          else
            qkv_chunk64(p, &tmC, &tmD, &tmE, stage, row, mb * BM + q * 32, nb * BN + ch * 32, v);
        }
      } else {
#pragma unroll 1
        for (int ch = chalf * (BN / 64); ch < (chalf + 1) * (BN / 64); ++ch) {
          float v[32];
          tmem_ld32(tbase + ch * 32, v);
          tmem_wait_ld();
          if constexpr (EPI == EPI_RESID) {
            resid_chunk(p, &tmC, stage, row, mb * BM + q * 32, nb * BN + ch * 32, v);
          } else if constexpr (EPI == EPI_STORE) {
            store_chunk(p, &tmC, stage, mb * BM + q * 32, nb * BN + ch * 32, v);
          } else {
            epilogue32<EPI>(p, row, nb * BN + ch * 32, v);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      // CTA-scope release: the arrival only orders this warp's TMEM reads
      // (tcgen05 fence above) before the MMAs that overwrite the accumulator.
      if (lane == 0) mbar_arrive_remote(tempty0 + acc * 8);  // the even CTA's barrier
    }
    // The staged stores and reductions must have completed before the CTA exits.
    if ((EPI == EPI_RESID || EPI == EPI_GELU || EPI == EPI_QKV || EPI == EPI_STORE) && lane == 0)
      bulk_wait_all();
  }

  tc_fence_before();
  __syncthreads();
  // Both CTAs must be done before the pair's TMEM is released and either leaves.
  cluster_sync();
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc_pair(tmem, TMEM_COLS);
  }
}

template <int EPI, bool WIDE>
cudaError_t launch_one(const CUtensorMap* tmA, const CUtensorMap* tmB, const CUtensorMap* tmC,
                       const CUtensorMap* tmD, const CUtensorMap* tmE, const GemmParams& p,
                       int max_ctas, cudaStream_t st) {
  static uint64_t set_up = 0;
  static int max_clusters_dev[64] = {};
  const size_t smem = GemmShape<WIDE>::SMEM;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.blockDim = dim3(320);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = once_per_device(&set_up, [&](int dev) {
    cudaError_t r = cudaFuncSetAttribute(gemm_tc_kernel<EPI, WIDE>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (r != cudaSuccess) return r;
    cfg.gridDim = dim3(2);
    int n = 0;
    r = cudaOccupancyMaxActiveClusters(&n, gemm_tc_kernel<EPI, WIDE>, &cfg);
    if (r != cudaSuccess) return r;
    if (n < 1) return cudaErrorInvalidConfiguration;
    max_clusters_dev[dev] = n;
    return cudaSuccess;
  });
  if (e != cudaSuccess) return e;
  int dev = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  const int max_clusters = max_clusters_dev[dev];
  const int n_m = (p.M + BM - 1) / BM, n_n = (p.N + GemmShape<WIDE>::BN - 1) / GemmShape<WIDE>::BN;
  const int n_pt = ((n_m + 1) / 2) * n_n;
  int clusters = max_clusters < n_pt ? max_clusters : n_pt;
  if (max_ctas >= 2 && clusters > max_ctas / 2) clusters = max_ctas / 2;
  cfg.gridDim = dim3(2 * clusters);
  cfg.numAttrs = 2;  // + programmatic stream serialization
  return cudaLaunchKernelEx(&cfg, gemm_tc_kernel<EPI, WIDE>, *tmA, *tmB, *tmC, *tmD, *tmE, p);
}

}  // namespace

size_t gemm_smem_bytes() {
  return GemmShape<true>::SMEM > GemmShape<false>::SMEM ? GemmShape<true>::SMEM : GemmShape<false>::SMEM;
}

// The wide tile pays off only where the main loop is long against the
// exposed epilogue: the down-projection (K = F).  Measured on the 1.3B wave:
// down 100 -> 94 us; QKV 66 -> 92, up 105 -> 130, out-projection 29 -> 31 us.
// It also halves the tile count, so it is taken only when its rounds of tiles
// over the clusters cost less: a wide tile's main loop is about twice a
// narrow one's, which TMA ingest stretches by ~1.22 (5B down-projection:
// 84 wide tiles on 76 clusters = 2 rounds, against 3 rounds of narrow ones).
bool use_wide(int epi, int M, int N, int K, int clusters) {
  if (epi != EPI_RESID || K < 4096) return false;
  if (clusters < 1) return true;
  const int n_mp = ((M + BM - 1) / BM + 1) / 2;
  const int rounds_w = (n_mp * ((N + 511) / 512) + clusters - 1) / clusters;
  const int rounds_n = (n_mp * ((N + 255) / 256) + clusters - 1) / clusters;
  return 2.0 * rounds_w <= 1.22 * rounds_n;
}

cudaError_t launch_gemm(int epi, const CUtensorMap* tmA, const CUtensorMap* tmB,
                        const CUtensorMap* tmC, const CUtensorMap* tmD, const CUtensorMap* tmE,
                        const GemmParams& p, int grid, cudaStream_t st) {
  if ((epi == EPI_RESID || epi == EPI_GELU || epi == EPI_STORE) && !tmC) return cudaErrorInvalidValue;
  if (epi == EPI_QKV && p.d % 64 == 0 && (!tmC || !tmD)) return cudaErrorInvalidValue;
  if (epi == EPI_QKV && p.vt_box && !tmE) return cudaErrorInvalidValue;
  const CUtensorMap* c = tmC ? tmC : tmA;  // unused by the other epilogues
  const CUtensorMap* dm = tmD ? tmD : tmA;
  const CUtensorMap* em = tmE ? tmE : tmA;
  const bool wide = use_wide(epi, p.M, p.N, p.K, grid / 2);
  switch (epi) {
    case EPI_QKV:
      return wide ? launch_one<EPI_QKV, true>(tmA, tmB, c, dm, em, p, grid, st)
                  : launch_one<EPI_QKV, false>(tmA, tmB, c, dm, em, p, grid, st);
    case EPI_RESID:
      return wide ? launch_one<EPI_RESID, true>(tmA, tmB, c, dm, em, p, grid, st)
                  : launch_one<EPI_RESID, false>(tmA, tmB, c, dm, em, p, grid, st);
    case EPI_GELU:
      return wide ? launch_one<EPI_GELU, true>(tmA, tmB, c, dm, em, p, grid, st)
                  : launch_one<EPI_GELU, false>(tmA, tmB, c, dm, em, p, grid, st);
    case EPI_EULER: return launch_one<EPI_EULER, false>(tmA, tmB, c, dm, em, p, grid, st);
    case EPI_STORE: return launch_one<EPI_STORE, false>(tmA, tmB, c, dm, em, p, grid, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace psv
