// Window attention of a chunk's queries over its own keys plus the still-noisy
// keys/values the W preceding chunks left at the same (block, step).
//
// The pages' dependency (AREX article "vLLM 与 Physis-AI 联合介绍 PhysisServe
// 推理系统", §难题; BAAI announcement "智源悟界·PhysisServe", Fig. 1): chunk c
// at step s reads the KV that chunk c-1 (and, with a window, chunks c-W..c-1)
// produced at the same step.  Those keys sit in a per-(stream, block, step)
// ring of W+1 slots; because every slot holds one of chunks c-W..c, the
// window is the ring prefix [0, kv_len) in physical slot order (softmax is
// invariant to key order).  No mask: a chunk is bidirectional.
//
// One CTA per (task, head, 128-query tile), warp-specialised:
//   warp 0      TMA: Q once, then K and V^T tiles of 128 keys (2 stages)
//   warp 1      TMEM allocator + MMA issuer: S = Q K^T into one of two TMEM
//               S buffers (S_{j+1} overlaps softmax j), O += P V into TMEM
//   warps 2..5  softmax, one query row per thread: online max/sum in the
//               log2 domain, lazy O rescale (only when the running max grows
//               by more than 8, i.e. a factor 256), P written as bf16 to
//               shared memory in the swizzled K-major layout the MMA reads.
#include "psv_device.cuh"
#include "psv_kernels.h"

namespace psv {

namespace {

constexpr int QT = 128;   // queries per CTA
constexpr int KT = 128;   // keys per tile
constexpr uint32_t TMEM_COLS = 512;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

template <int DH>
struct AttnCfg {
  static constexpr int AW = DH < 64 ? DH : 64;          // elements per swizzle row
  static constexpr int ROWB = AW * 2;                   // bytes per swizzle row
  static constexpr int NA = DH / AW;                    // atoms along dh
  static constexpr int Q_BYTES = QT * DH * 2;
  static constexpr int K_BYTES = KT * DH * 2;
  static constexpr int V_BYTES = DH * KT * 2;           // V^T tile [DH][128 keys]
  static constexpr int P_BYTES = QT * KT * 2;
  static constexpr int Q_ATOM = QT * ROWB;
  static constexpr int K_ATOM = KT * ROWB;
  static constexpr int V_ATOM = DH * 128;               // [DH rows][64 keys]
  static constexpr int P_ATOM = QT * 128;               // [128 rows][64 keys]
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + Q_BYTES;
  static constexpr int OFF_V = OFF_K + 2 * K_BYTES;
  static constexpr int OFF_P = OFF_V + 2 * V_BYTES;
  static constexpr int OFF_BAR = OFF_P + P_BYTES;
  static constexpr int N_BARS = 12;
  static constexpr size_t SMEM = 1024 + OFF_BAR + N_BARS * 8 + 16;
};

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, int* err) {
  int ok = 0;
  if (lane_id() == 0) ok = mbar_wait(bar, parity, err, ERR_ATTN_TIMEOUT) ? 1 : 0;
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

template <int DH>
__global__ void __launch_bounds__(192, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tmQ,
                   const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const AttnParams p) {
  using Cfg = AttnCfg<DH>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem + Cfg::OFF_Q;
  uint8_t* sK = smem + Cfg::OFF_K;
  uint8_t* sV = smem + Cfg::OFF_V;
  uint8_t* sP = smem + Cfg::OFF_P;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Cfg::OFF_BAR);
  uint64_t* q_full = bars + 0;
  uint64_t* kv_full = bars + 1;   // [2]
  uint64_t* kv_empty = bars + 3;  // [2]
  uint64_t* s_full = bars + 5;    // [2]
  uint64_t* s_empty = bars + 7;   // [2]
  uint64_t* p_full = bars + 9;
  uint64_t* o_done = bars + 10;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + Cfg::N_BARS);

  const int warp = warp_id(), lane = lane_id();
  const int work = blockIdx.x;
  const int qt = work % p.n_qtiles;
  const int head = (work / p.n_qtiles) % p.H;
  const int ti = work / (p.n_qtiles * p.H);
  const TaskDev task = p.tasks[ti];
  const int ring = task.ring0 + p.block * p.S;
  const int kv_len = task.kv_len;
  const int nT = (kv_len + KT - 1) / KT;
  const int qrow0 = task.row0 + qt * QT;  // first query row in the wave batch

  if (warp == 0 && lane == 0) {
    for (int i = 0; i < Cfg::N_BARS; ++i) mbar_init(&bars[i], (i == 7 || i == 8 || i == 9) ? 4 : 1);
    fence_mbar_init();
    prefetch_tensormap(&tmQ);
    prefetch_tensormap(&tmK);
    prefetch_tensormap(&tmV);
  }
  if (warp == 1) tmem_alloc(tmem_slot, TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tmem_o = tmem + 2 * KT;  // O accumulator columns [256, 256 + DH)

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer
      int issued = 0;
      bool ok = true;
      mbar_arrive_expect_tx(q_full, Cfg::Q_BYTES);
#pragma unroll
      for (int a = 0; a < Cfg::NA; ++a)
        tma_load_2d(sQ + a * Cfg::Q_ATOM, &tmQ, q_full, head * DH + a * Cfg::AW, qrow0);
      for (int j = 0; j < nT; ++j) {
        const int st = j & 1;
        const uint32_t use = j >> 1;
        if (!mbar_wait(&kv_empty[st], (use & 1) ^ 1, p.err, ERR_ATTN_TIMEOUT)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&kv_full[st], Cfg::K_BYTES + Cfg::V_BYTES);
        uint8_t* k_dst = sK + st * Cfg::K_BYTES;
        uint8_t* v_dst = sV + st * Cfg::V_BYTES;
#pragma unroll
        for (int a = 0; a < Cfg::NA; ++a)
          tma_load_3d(k_dst + a * Cfg::K_ATOM, &tmK, &kv_full[st], head * DH + a * Cfg::AW,
                      j * KT, ring);
#pragma unroll
        for (int a = 0; a < 2; ++a)
          tma_load_3d(v_dst + a * Cfg::V_ATOM, &tmV, &kv_full[st], j * KT + a * 64, 0,
                      ring * p.H + head);
        ++issued;
      }
      if (!ok || error_raised(p.err)) {
        const uint64_t t0 = global_timer_ns();
        while (!mbar_try_wait(q_full, 0) && global_timer_ns() - t0 < kWaitLimitNs) {
        }
        for (int j = (issued > 2 ? issued - 2 : 0); j < issued; ++j) {
          while (!mbar_try_wait(&kv_full[j & 1], (j >> 1) & 1) &&
                 global_timer_ns() - t0 < kWaitLimitNs) {
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer
      constexpr uint32_t IDESC_S = umma_idesc_bf16(QT, KT);
      constexpr uint32_t IDESC_O = umma_idesc_bf16(QT, DH);
      auto issue_s = [&](int j) {
        const int st = j & 1;
        const uint32_t q0 = smem_u32(sQ), k0 = smem_u32(sK + st * Cfg::K_BYTES);
#pragma unroll
        for (int kk = 0; kk < DH / 16; ++kk) {
          const int e = kk * 16;
          const uint32_t off_q = (e / Cfg::AW) * Cfg::Q_ATOM + (e % Cfg::AW) * 2;
          const uint32_t off_k = (e / Cfg::AW) * Cfg::K_ATOM + (e % Cfg::AW) * 2;
          umma_bf16(tmem + st * KT, umma_desc_kmajor(q0 + off_q, Cfg::ROWB),
                    umma_desc_kmajor(k0 + off_k, Cfg::ROWB), IDESC_S, kk != 0);
        }
        umma_commit(&s_full[st]);
      };
      bool ok = mbar_wait(q_full, 0, p.err, ERR_ATTN_TIMEOUT);
      if (ok) ok = mbar_wait(&kv_full[0], 0, p.err, ERR_ATTN_TIMEOUT);
      if (ok) {
        tc_fence_after();
        issue_s(0);
      }
      for (int j = 0; j < nT && ok; ++j) {
        if (j + 1 < nT) {
          const int st1 = (j + 1) & 1;
          const uint32_t use1 = (j + 1) >> 1;
          if (!mbar_wait(&kv_full[st1], use1 & 1, p.err, ERR_ATTN_TIMEOUT) ||
              !mbar_wait(&s_empty[st1], (use1 & 1) ^ 1, p.err, ERR_ATTN_TIMEOUT)) {
            ok = false;
            break;
          }
          tc_fence_after();
          issue_s(j + 1);
        }
        if (!mbar_wait(p_full, j & 1, p.err, ERR_ATTN_TIMEOUT)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t p0 = smem_u32(sP), v0 = smem_u32(sV + (j & 1) * Cfg::V_BYTES);
#pragma unroll
        for (int kk = 0; kk < KT / 16; ++kk) {
          const uint32_t off_p = (kk >> 2) * Cfg::P_ATOM + (kk & 3) * 32;
          const uint32_t off_v = (kk >> 2) * Cfg::V_ATOM + (kk & 3) * 32;
          umma_bf16(tmem_o, umma_desc_kmajor(p0 + off_p, 128), umma_desc_kmajor(v0 + off_v, 128),
                    IDESC_O, (j | kk) != 0);
        }
        umma_commit(&kv_empty[j & 1]);
        umma_commit(o_done);
      }
    }
  } else {
    // ---------------- softmax warps: thread = query row r of the tile
    const int q = warp & 3;
    const int r = q * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
    const float sl2 = p.scale_log2;
    float m = -INFINITY, l = 0.0f;
    bool ok = true;
    for (int j = 0; j < nT; ++j) {
      const int st = j & 1;
      if (!warp_wait(&s_full[st], (j >> 1) & 1, p.err)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float s[KT];
#pragma unroll
      for (int c = 0; c < KT / 32; ++c) tmem_ld32(tmem + st * KT + c * 32 + lane_off, s + c * 32);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s_empty[st]);

      const int key0 = j * KT;
      if (key0 + KT > kv_len) {
#pragma unroll
        for (int c = 0; c < KT; ++c)
          if (key0 + c >= kv_len) s[c] = -INFINITY;
      }
      float mx = s[0];
#pragma unroll
      for (int c = 1; c < KT; ++c) mx = fmaxf(mx, s[c]);
      const float m_tile = mx * sl2;

      if (j > 0) {
        if (!warp_wait(o_done, (j - 1) & 1, p.err)) {
          ok = false;
          break;
        }
        tc_fence_after();
      }
      const bool grow = m_tile > m + kRescaleThreshold;
      if (__any_sync(0xffffffffu, grow)) {
        const float m_new = grow ? m_tile : m;
        const float alpha = grow ? fast_exp2(m - m_new) : 1.0f;
        if (j > 0) {
#pragma unroll 1
          for (int c = 0; c < DH / 32; ++c) {
            float o[32];
            tmem_ld32(tmem_o + c * 32 + lane_off, o);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] *= alpha;
            tmem_st32(tmem_o + c * 32 + lane_off, o);
          }
          tmem_wait_st();
        }
        l *= alpha;
        m = m_new;
      }
      // P = exp2(s * scale_log2 - m), row sum, bf16 into the swizzled tile.
      float sum = 0.0f;
      uint8_t* prow = sP + r * 128;
#pragma unroll
      for (int cidx = 0; cidx < KT / 8; ++cidx) {
        float pv[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          pv[i] = fast_exp2(fmaf(s[cidx * 8 + i], sl2, -m));
          sum += pv[i];
        }
        uint4 w;
        w.x = pack_bf16x2(pv[0], pv[1]);
        w.y = pack_bf16x2(pv[2], pv[3]);
        w.z = pack_bf16x2(pv[4], pv[5]);
        w.w = pack_bf16x2(pv[6], pv[7]);
        const int atom = cidx >> 3, chunk = cidx & 7;
        *reinterpret_cast<uint4*>(prow + atom * Cfg::P_ATOM + ((chunk ^ (r & 7)) << 4)) = w;
      }
      l += sum;
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full);
    }
    if (ok && warp_wait(o_done, (nT - 1) & 1, p.err)) {
      tc_fence_after();
      const bool valid = (qt * QT + r) < p.T;
      const float inv_l = 1.0f / l;
      __nv_bfloat16* dst = p.o + static_cast<int64_t>(qrow0 + r) * p.d + head * DH;
#pragma unroll 1
      for (int c = 0; c < DH / 32; ++c) {
        float o[32];
        tmem_ld32(tmem_o + c * 32 + lane_off, o);
        tmem_wait_ld();
        if (valid) {
          uint4* d4 = reinterpret_cast<uint4*>(dst + c * 32);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            uint4 w;
            w.x = pack_bf16x2(o[8 * i + 0] * inv_l, o[8 * i + 1] * inv_l);
            w.y = pack_bf16x2(o[8 * i + 2] * inv_l, o[8 * i + 3] * inv_l);
            w.z = pack_bf16x2(o[8 * i + 4] * inv_l, o[8 * i + 5] * inv_l);
            w.w = pack_bf16x2(o[8 * i + 6] * inv_l, o[8 * i + 7] * inv_l);
            d4[i] = w;
          }
        }
      }
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

template <int DH>
cudaError_t launch_dh(const CUtensorMap* tmQ, const CUtensorMap* tmK, const CUtensorMap* tmV,
                      const AttnParams& p, int n_tasks, cudaStream_t st) {
  static bool attr_set = false;
  // Every variant asks for more than half the SM's shared memory so that one
  // CTA holds an SM: the 512 TMEM columns it allocates are then always free.
  const size_t smem = attn_smem_bytes(DH);
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel<DH>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const int grid = n_tasks * p.H * p.n_qtiles;
  attn_tc_kernel<DH><<<grid, 192, smem, st>>>(*tmQ, *tmK, *tmV, p);
  return cudaGetLastError();
}

}  // namespace

size_t attn_smem_bytes(int dh) {
  size_t need = 0;
  switch (dh) {
    case 32: need = AttnCfg<32>::SMEM; break;
    case 64: need = AttnCfg<64>::SMEM; break;
    default: need = AttnCfg<128>::SMEM; break;
  }
  const size_t one_per_sm = 120 * 1024;
  return need > one_per_sm ? need : one_per_sm;
}

cudaError_t launch_attention(const CUtensorMap* tmQ, const CUtensorMap* tmK,
                             const CUtensorMap* tmV, const AttnParams& p, int n_tasks,
                             cudaStream_t st) {
  switch (p.dh) {
    case 32: return launch_dh<32>(tmQ, tmK, tmV, p, n_tasks, st);
    case 64: return launch_dh<64>(tmQ, tmK, tmV, p, n_tasks, st);
    case 128: return launch_dh<128>(tmQ, tmK, tmV, p, n_tasks, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace psv
