// Persistent tcgen05 GEMM with fused epilogues:  C = A W^T + bias.
//
// A [M, K] bf16 activations and W [N, K] bf16 weights (nn.Linear layout)
// are both K-major, so TMA loads 128-byte-swizzled tiles that feed
// tcgen05.mma directly.  One CTA per SM, warp-specialised:
//   warp 0      TMA producer (4-stage smem ring, 48 KB per stage)
//   warp 1      TMEM allocator + single-thread MMA issuer (128x256x16 MMAs)
//   warps 2..9  epilogue: tcgen05.ld of a 128x256 f32 accumulator (double
//               buffered in TMEM, 2 x 256 columns) and the fused epilogue;
//               two warps per TMEM lane quadrant, each taking 128 columns.
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

constexpr int BM = kGemmBM, BN = kGemmBN, BK = kGemmBK, STAGES = kGemmStages;
constexpr int A_BYTES = BM * BK * 2;  // 16 KB
constexpr int B_BYTES = BN * BK * 2;  // 32 KB
constexpr uint32_t TMEM_COLS = 512;   // two 256-column accumulators
constexpr uint32_t IDESC = umma_idesc_bf16(BM, BN);

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

// Fused epilogue of 32 consecutive columns [n0, n0+32) of one row.
template <int EPI>
__device__ __forceinline__ void epilogue32(const GemmParams& p, int row, int n0, float* v) {
  if (row >= p.M || n0 >= p.N) return;
  const int ti = row / p.T;
  const TaskDev& t = p.tasks[ti];
  const int li = row - t.row0;  // token index within the chunk

  if (EPI == EPI_EULER) {
    // Velocity head: x += dt * (acc + b_out); only the first C columns exist.
    float* x = p.state + (static_cast<int64_t>(t.state_slot) * p.T + li) * p.C;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const int n = n0 + i;
      if (n < p.N) x[n] += t.dt * (v[i] + p.bias[n]);
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

  if (EPI == EPI_GELU) {
    uint4* dst = reinterpret_cast<uint4*>(p.u + static_cast<int64_t>(row) * p.N + n0);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint4 w;
      w.x = pack_bf16x2(gelu_tanh(v[8 * i + 0]), gelu_tanh(v[8 * i + 1]));
      w.y = pack_bf16x2(gelu_tanh(v[8 * i + 2]), gelu_tanh(v[8 * i + 3]));
      w.z = pack_bf16x2(gelu_tanh(v[8 * i + 4]), gelu_tanh(v[8 * i + 5]));
      w.w = pack_bf16x2(gelu_tanh(v[8 * i + 6]), gelu_tanh(v[8 * i + 7]));
      dst[i] = w;
    }
  } else if (EPI == EPI_RESID) {
    const float4* g4 = reinterpret_cast<const float4*>(
        p.mod + t.mod0 + static_cast<int64_t>(p.block) * 6 * p.d + p.gate_off + n0);
    float4* h4 = reinterpret_cast<float4*>(p.h + static_cast<int64_t>(row) * p.d + n0);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float4 g = __ldg(g4 + i);
      float4 hv = h4[i];
      hv.x += g.x * v[4 * i];
      hv.y += g.y * v[4 * i + 1];
      hv.z += g.z * v[4 * i + 2];
      hv.w += g.w * v[4 * i + 3];
      h4[i] = hv;
    }
  } else if (EPI == EPI_QKV) {
    const int sec = n0 / p.d;  // 0 = q, 1 = k, 2 = v
    const int j0 = n0 - sec * p.d;
    const int head = j0 / p.dh;
    const int e0 = j0 - head * p.dh;
    const int half = p.dh >> 1;
    if (sec < 2) {
      // Rotate pairs (e, e+1) by angle (c*T + li) * f_{e/2}; the angle is
      // assembled from two tables built in f64 on the host.
      const float2* rb = p.rope_base + static_cast<int64_t>(t.rope_slot) * half + (e0 >> 1);
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

// Warp-uniform bounded wait: lane 0 polls, the verdict is broadcast.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, int* err, int code) {
  int ok = 0;
  if (lane_id() == 0) ok = mbar_wait(bar, parity, err, code) ? 1 : 0;
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

template <int EPI>
__global__ void __launch_bounds__(320, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA,
                   const __grid_constant__ CUtensorMap tmB, const GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * A_BYTES;
  uint64_t* full = reinterpret_cast<uint64_t*>(sB + STAGES * B_BYTES);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tempty + 2);

  const int warp = warp_id(), lane = lane_id();
  const int n_m = (p.M + BM - 1) / BM;
  const int n_n = (p.N + BN - 1) / BN;
  const int n_tiles = n_m * n_n;
  const int nk = (p.K + BK - 1) / BK;

  if (warp == 0 && lane == 0) {
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tfull[i], 1);
      mbar_init(&tempty[i], 8);
    }
    fence_mbar_init();
    prefetch_tensormap(&tmA);
    prefetch_tensormap(&tmB);
  }
  if (warp == 1) tmem_alloc(tmem_slot, TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer
      int it = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x) {
        const int mb = tile % n_m, nb = tile / n_m;
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int st = it % STAGES;
          const uint32_t ph = (it / STAGES) & 1;
          if (!mbar_wait(&empty[st], ph ^ 1, p.err, ERR_GEMM_TIMEOUT)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[st], A_BYTES + B_BYTES);
          tma_load_2d(sA + st * A_BYTES, &tmA, &full[st], kb * BK, mb * BM);
          tma_load_3d(sB + st * B_BYTES, &tmB, &full[st], kb * BK, nb * BN, p.wz);
        }
      }
      if (!ok || error_raised(p.err)) {
        // Error path: let the loads already issued land before the CTA exits.
        const uint64_t t0 = global_timer_ns();
        for (int j = (it > STAGES ? it - STAGES : 0); j < it; ++j) {
          while (!mbar_try_wait(&full[j % STAGES], (j / STAGES) & 1)) {
            if (global_timer_ns() - t0 > kWaitLimitNs) break;
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer
      int it = 0, tc = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x, ++tc) {
        const int acc = tc & 1;
        const uint32_t aph = (tc >> 1) & 1;
        if (!mbar_wait(&tempty[acc], aph ^ 1, p.err, ERR_GEMM_TIMEOUT)) break;
        tc_fence_after();
        const uint32_t dtm = tmem + acc * BN;
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int st = it % STAGES;
          const uint32_t ph = (it / STAGES) & 1;
          if (!mbar_wait(&full[st], ph, p.err, ERR_GEMM_TIMEOUT)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(sA + st * A_BYTES);
          const uint32_t b0 = smem_u32(sB + st * B_BYTES);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k) {
            umma_bf16(dtm, umma_desc_kmajor(a0 + k * 32, 128), umma_desc_kmajor(b0 + k * 32, 128),
                      IDESC, (kb | k) != 0);
          }
          umma_commit(&empty[st]);
        }
        if (ok) umma_commit(&tfull[acc]);
      }
    }
  } else {
    // ---------------- epilogue warps (TMEM lane quadrant = warp % 4)
    const int q = warp & 3;
    const int chalf = (warp - 2) >> 2;  // which 128 accumulator columns
    int tc = 0;
    for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x, ++tc) {
      const int mb = tile % n_m, nb = tile / n_m;
      const int acc = tc & 1;
      const uint32_t aph = (tc >> 1) & 1;
      if (!warp_wait(&tfull[acc], aph, p.err, ERR_GEMM_TIMEOUT)) break;
      tc_fence_after();
      const int row = mb * BM + q * 32 + lane;
      const uint32_t tbase = tmem + acc * BN + (static_cast<uint32_t>(q * 32) << 16);
#pragma unroll 1
      for (int ch = chalf * (BN / 64); ch < (chalf + 1) * (BN / 64); ++ch) {
        float v[32];
        tmem_ld32(tbase + ch * 32, v);
        tmem_wait_ld();
        epilogue32<EPI>(p, row, nb * BN + ch * 32, v);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[acc]);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

template <int EPI>
cudaError_t launch_one(const CUtensorMap* tmA, const CUtensorMap* tmB, const GemmParams& p,
                       int grid, cudaStream_t st) {
  static bool attr_set = false;
  const size_t smem = gemm_smem_bytes();
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(gemm_tc_kernel<EPI>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  gemm_tc_kernel<EPI><<<grid, 320, smem, st>>>(*tmA, *tmB, p);
  return cudaGetLastError();
}

}  // namespace

size_t gemm_smem_bytes() {
  return 1024 + STAGES * (A_BYTES + B_BYTES) + (2 * STAGES + 4) * sizeof(uint64_t) + 16;
}

cudaError_t launch_gemm(int epi, const CUtensorMap* tmA, const CUtensorMap* tmB,
                        const GemmParams& p, int grid, cudaStream_t st) {
  switch (epi) {
    case EPI_QKV: return launch_one<EPI_QKV>(tmA, tmB, p, grid, st);
    case EPI_RESID: return launch_one<EPI_RESID>(tmA, tmB, p, grid, st);
    case EPI_GELU: return launch_one<EPI_GELU>(tmA, tmB, p, grid, st);
    case EPI_EULER: return launch_one<EPI_EULER>(tmA, tmB, p, grid, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace psv
