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
// One CTA per (task, head, pair of 128-query tiles); both query tiles share
// every K / V^T tile loaded.  Warp roles (320 threads):
//   warp 0      TMA: Q0, Q1 once, then K tiles of 128 keys (2 stages)
//   warp 18     TMA: V^T tiles (2 stages).  K and V stages are released
//               separately (K after both S MMAs, V after both P.V MMAs), so
//               the next K tile streams in a whole tile ahead of its use
//   warp 1      TMEM allocator + MMA issuer, per key tile j:
//                 PV0_j, S0_{j+1}, PV1_j, S1_{j+1}
//               so the tensor core always has the other tile's work while a
//               softmax warpgroup runs (ping-pong)
//   warps 2..9  softmax of query tile 0, warps 10..17 of tile 1: two threads
//               per query row (warps w and w+4 share a TMEM lane quadrant and
//               take 64 of the 128 keys each; the row max is exchanged through
//               shared memory); online max/sum in the log2 domain, lazy O
//               rescale (only when the running max grows by more than 2^8), P
//               in bf16 written to TMEM over the S columns (keys [64h, 64h+64)
//               to packed columns [64h, 64h+32)) and consumed by the P.V MMA
//               straight from TMEM.  S is read twice (max pass, exp pass) to
//               stay within the 96 registers 18 warps allow.
// TMEM columns: S0/P0 [0,128), S1/P1 [128,256), O0 [256,256+dh), O1 [384,..).
// Long windows (>= 16 key tiles) are split into two fixed halves handled by
// two CTAs, so that a wave's few hundred equal work units spread evenly over
// the SMs; each half leaves its unnormalised O, m and l in a partial area and
// the CTA that arrives second on the pair's counter merges both in a fixed
// order (half 0, half 1), so the result does not depend on which finished
// first.
// tcgen05 MMAs of one issuing thread execute in order, so S_{i,j+1} (issued
// after PV_{i,j}) only overwrites P_{i,j} once it was consumed, and when
// S_{i,j+1} is complete O_i is stable for the softmax warps to rescale.
#include "psv_device.cuh"
#include "psv_kernels.h"

namespace psv {

namespace {

constexpr int QT = 128;   // queries per tile (two tiles per CTA)
constexpr int KT = 128;   // keys per tile
constexpr uint32_t TMEM_COLS = 512;
constexpr float kRescaleThreshold = 8.0f;  // log2 units
#ifndef ATTN_K_STAGES
#define ATTN_K_STAGES 3
#endif
#ifndef ATTN_V_STAGES
#define ATTN_V_STAGES 2
#endif
constexpr int kThreads = 608;  // Q/K TMA warp, MMA warp, 2 x 8 softmax warps, V TMA warp

template <int DH>
struct AttnCfg {
  static constexpr int AW = DH < 64 ? DH : 64;  // elements per swizzle row
  static constexpr int ROWB = AW * 2;           // bytes per swizzle row
  static constexpr int NA = DH / AW;            // atoms along dh
  static constexpr int Q_BYTES = QT * DH * 2;
  static constexpr int K_BYTES = KT * DH * 2;
  static constexpr int V_BYTES = DH * KT * 2;   // V^T tile [DH][128 keys]
  static constexpr int Q_ATOM = QT * ROWB;
  static constexpr int K_ATOM = KT * ROWB;
  static constexpr int V_ATOM = DH * 128;       // [DH rows][64 keys]
  static constexpr int KS = ATTN_K_STAGES;      // K tile stages
  static constexpr int VS = ATTN_V_STAGES;      // V^T tile stages
  static constexpr int OFF_Q = 0;               // two query tiles
  static constexpr int OFF_K = OFF_Q + 2 * Q_BYTES;
  static constexpr int OFF_V = OFF_K + KS * K_BYTES;
  static constexpr int OFF_BAR = OFF_V + VS * V_BYTES;
  static constexpr int N_BARS = 1 + 2 * KS + 2 * VS + 6;
  // barriers, the TMEM address word, then the row-max / row-sum exchange
  // area [2 query tiles][2 key halves][128 rows] f32
  // The dynamic shared-memory window starts 1024-byte aligned (the kernel
  // has no static shared variables; it checks the alignment at run time).
  static constexpr size_t SMEM = OFF_BAR + N_BARS * 8 + 16 + 2 * 2 * QT * 4;
  static constexpr int OH = DH / 2;                 // O columns per thread
  static constexpr int OC = OH < 32 ? OH : 32;      // O columns per TMEM access
};

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, int* err) {
  int ok = 0;
  if (lane_id() == 0) ok = mbar_wait(bar, parity, err, ERR_ATTN_TIMEOUT) ? 1 : 0;
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// D(tmem) (+)= A(tmem, bf16 packed 2 per column) x B(smem descriptor).
__device__ __forceinline__ void umma_bf16_tmem_a(uint32_t tmem_d, uint32_t tmem_a, uint64_t bdesc,
                                                 uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(tmem_d),
      "r"(tmem_a), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
      "r"(v[15])
      : "memory");
}

__device__ __forceinline__ void tmem_ld16f(uint32_t taddr, float* v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// O-column access of OC (16 or 32) f32 columns.
template <int OC>
__device__ __forceinline__ void o_ld(uint32_t taddr, float* v) {
  if constexpr (OC == 32) tmem_ld32(taddr, v);
  else tmem_ld16f(taddr, v);
}
template <int OC>
__device__ __forceinline__ void o_st(uint32_t taddr, const float* v) {
  if constexpr (OC == 32) {
    tmem_st32(taddr, v);
  } else {
    uint32_t u[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) u[e] = __float_as_uint(v[e]);
    tmem_st16(taddr, u);
  }
}

__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// (x0, x1) * s + (b, b) on the packed f32x2 path.
__device__ __forceinline__ void ffma2(float& x0, float& x1, float s, float b) {
  uint64_t x, sv, bv;
  asm("mov.b64 %0, {%1, %2};" : "=l"(x) : "f"(x0), "f"(x1));
  asm("mov.b64 %0, {%1, %1};" : "=l"(sv) : "f"(s));
  asm("mov.b64 %0, {%1, %1};" : "=l"(bv) : "f"(b));
  asm("fma.rn.f32x2 %0, %0, %1, %2;" : "+l"(x) : "l"(sv), "l"(bv));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(x0), "=f"(x1) : "l"(x));
}

__device__ __forceinline__ void fadd2(float& a0, float& a1, float b0, float b1) {
  uint64_t a, b;
  asm("mov.b64 %0, {%1, %2};" : "=l"(a) : "f"(a0), "f"(a1));
  asm("mov.b64 %0, {%1, %2};" : "=l"(b) : "f"(b0), "f"(b1));
  asm("add.f32x2 %0, %0, %1;" : "+l"(a) : "l"(b));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a0), "=f"(a1) : "l"(a));
}

template <int DH>
__global__ void __launch_bounds__(kThreads, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tmQ,
                   const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const AttnParams p) {
  using Cfg = AttnCfg<DH>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw;
  if (smem_u32(smem) & 1023) {  // swizzled TMA tiles need 1024-byte alignment
    if (threadIdx.x == 0) raise_error(p.err, ERR_BOUNDS);
    return;
  }
  uint8_t* sQ = smem + Cfg::OFF_Q;
  uint8_t* sK = smem + Cfg::OFF_K;
  uint8_t* sV = smem + Cfg::OFF_V;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Cfg::OFF_BAR);
  constexpr int KS = Cfg::KS, VS = Cfg::VS;
  uint64_t* q_full = bars + 0;
  uint64_t* s_full = bars + 1;             // [2] query tile
  uint64_t* p_full = bars + 3;             // [2] query tile (8 warps arrive)
  uint64_t* o_done = bars + 5;             // [2] query tile
  uint64_t* k_full = bars + 7;             // [KS] stage
  uint64_t* k_empty = k_full + KS;         // [KS] stage: K tile consumed by both S MMAs
  uint64_t* v_full = k_empty + KS;         // [VS] stage
  uint64_t* v_empty = v_full + VS;         // [VS] stage: V tile consumed by both P.V MMAs
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + Cfg::N_BARS);
  int* s_last_p = reinterpret_cast<int*>(tmem_slot + 1);

  const int warp = warp_id(), lane = lane_id();
  // Work item -> (task, head, query pair, key half), grouped by (task, head)
  // so that the CTAs sharing K/V (every query pair and key half of the
  // group) run together while their K/V is L2-resident.
  const int n_pairs = (p.T + 2 * QT - 1) / (2 * QT);
  int ti = 0, head = 0, pair = 0, half = 0, nsplit = 1;
  {
    int idx = blockIdx.x;
    for (int t = 0; t < p.n_tasks; ++t) {
      const int ns = ((p.tasks[t].kv_len + KT - 1) / KT >= kAttnSplitMinTiles) ? 2 : 1;
      const int cnt = p.H * n_pairs * ns;
      if (idx < cnt) {
        ti = t, nsplit = ns, half = idx % ns, pair = (idx / ns) % n_pairs, head = idx / (ns * n_pairs);
        break;
      }
      idx -= cnt;
    }
  }
  const TaskDev task = p.tasks[ti];
  const int ring = task.ring0 + p.block * p.S;
  const int kv_len = task.kv_len;
  const int nT_all = (kv_len + KT - 1) / KT;
  const int j_begin = (half == 0) ? 0 : nT_all / 2;
  const int j_end = (nsplit == 1 || half == 1) ? nT_all : nT_all / 2;
  const int nT = j_end - j_begin;  // key tiles of this CTA: [j_begin, j_end)
  const int qrow0 = task.row0 + pair * 2 * QT;  // first query row in the wave batch
  const bool has_q1 = pair * 2 * QT + QT < p.T;
  const int item = (ti * p.H + head) * p.max_pairs + pair;

  if (warp == 0 && lane == 0) {
    for (int i = 0; i < Cfg::N_BARS; ++i) mbar_init(&bars[i], (i == 3 || i == 4) ? 8 : 1);
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

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer
      int issued = 0;
      bool ok = true;
      mbar_arrive_expect_tx(q_full, Cfg::Q_BYTES * (has_q1 ? 2 : 1));
#pragma unroll
      for (int a = 0; a < Cfg::NA; ++a)
        tma_load_2d(sQ + a * Cfg::Q_ATOM, &tmQ, q_full, head * DH + a * Cfg::AW, qrow0);
      if (has_q1) {
#pragma unroll
        for (int a = 0; a < Cfg::NA; ++a)
          tma_load_2d(sQ + Cfg::Q_BYTES + a * Cfg::Q_ATOM, &tmQ, q_full, head * DH + a * Cfg::AW,
                      qrow0 + QT);
      }
      for (int j = 0; j < nT; ++j) {
        const int st = j % KS;
        const uint32_t use = j / KS;
        if (!mbar_wait(&k_empty[st], (use & 1) ^ 1, p.err, ERR_ATTN_TIMEOUT)) {
          ok = false;
          break;
        }
        uint8_t* k_dst = sK + st * Cfg::K_BYTES;
        mbar_arrive_expect_tx(&k_full[st], Cfg::K_BYTES);
#pragma unroll
        for (int a = 0; a < Cfg::NA; ++a)
          tma_load_3d(k_dst + a * Cfg::K_ATOM, &tmK, &k_full[st], head * DH + a * Cfg::AW,
                      (j_begin + j) * KT, ring);
        ++issued;
      }
      if (!ok || error_raised(p.err)) {
        // Error path: let the loads already issued land before the CTA exits.
        const uint64_t t0 = global_timer_ns();
        while (!mbar_try_wait(q_full, 0) && global_timer_ns() - t0 < kWaitLimitNs) {
        }
        for (int j = (issued > KS ? issued - KS : 0); j < issued; ++j) {
          while (!mbar_try_wait(&k_full[j % KS], (j / KS) & 1) &&
                 global_timer_ns() - t0 < kWaitLimitNs) {
          }
        }
      }
    }
  } else if (warp == kThreads / 32 - 1) {
    if (lane == 0) {
      // ---------------- V^T producer (own warp, so K loads run ahead of V)
      int issued = 0;
      bool ok = true;
      for (int j = 0; j < nT; ++j) {
        const int st = j % VS;
        const uint32_t use = j / VS;
        if (!mbar_wait(&v_empty[st], (use & 1) ^ 1, p.err, ERR_ATTN_TIMEOUT)) {
          ok = false;
          break;
        }
        uint8_t* v_dst = sV + st * Cfg::V_BYTES;
        mbar_arrive_expect_tx(&v_full[st], Cfg::V_BYTES);
#pragma unroll
        for (int a = 0; a < 2; ++a)
          tma_load_3d(v_dst + a * Cfg::V_ATOM, &tmV, &v_full[st], (j_begin + j) * KT + a * 64, 0,
                      ring * p.H + head);
        ++issued;
      }
      if (!ok || error_raised(p.err)) {
        const uint64_t t0 = global_timer_ns();
        for (int j = (issued > VS ? issued - VS : 0); j < issued; ++j) {
          while (!mbar_try_wait(&v_full[j % VS], (j / VS) & 1) &&
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
      auto issue_s = [&](int i, int j) {
        const uint32_t q0 = smem_u32(sQ + i * Cfg::Q_BYTES);
        const uint32_t k0 = smem_u32(sK + (j % KS) * Cfg::K_BYTES);
#pragma unroll
        for (int kk = 0; kk < DH / 16; ++kk) {
          const int e = kk * 16;
          const uint32_t off_q = (e / Cfg::AW) * Cfg::Q_ATOM + (e % Cfg::AW) * 2;
          const uint32_t off_k = (e / Cfg::AW) * Cfg::K_ATOM + (e % Cfg::AW) * 2;
          umma_bf16(tmem + i * KT, umma_desc_kmajor(q0 + off_q, Cfg::ROWB),
                    umma_desc_kmajor(k0 + off_k, Cfg::ROWB), IDESC_S, kk != 0);
        }
        umma_commit(&s_full[i]);
      };
      auto issue_pv = [&](int i, int j) {
        const uint32_t v0 = smem_u32(sV + (j % VS) * Cfg::V_BYTES);
#pragma unroll
        for (int kk = 0; kk < KT / 16; ++kk) {
          const uint32_t off_v = (kk >> 2) * Cfg::V_ATOM + (kk & 3) * 32;
          // keys [64h, 64h+64) of P sit in packed columns [64h, 64h+32) of S_i
          umma_bf16_tmem_a(tmem + 2 * KT + i * 128, tmem + i * KT + (kk >> 2) * 64 + (kk & 3) * 8,
                           umma_desc_kmajor(v0 + off_v, 128), IDESC_O, (j | kk) != 0);
        }
        umma_commit(&o_done[i]);
      };
      bool ok = mbar_wait(q_full, 0, p.err, ERR_ATTN_TIMEOUT) &&
                mbar_wait(&k_full[0], 0, p.err, ERR_ATTN_TIMEOUT);
      if (ok) {
        tc_fence_after();
        issue_s(0, 0);
        if (has_q1) issue_s(1, 0);
        umma_commit(&k_empty[0]);
      }
      for (int j = 0; j < nT && ok; ++j) {
        const int vst = j % VS;
        const bool next = j + 1 < nT;
        if (!mbar_wait(&p_full[0], j & 1, p.err, ERR_ATTN_TIMEOUT) ||
            !mbar_wait(&v_full[vst], (j / VS) & 1, p.err, ERR_ATTN_TIMEOUT)) {
          ok = false;
          break;
        }
        tc_fence_after();
        issue_pv(0, j);
        if (next) {
          if (!mbar_wait(&k_full[(j + 1) % KS], ((j + 1) / KS) & 1, p.err, ERR_ATTN_TIMEOUT)) {
            ok = false;
            break;
          }
          tc_fence_after();
          issue_s(0, j + 1);
        }
        if (has_q1) {
          if (!mbar_wait(&p_full[1], j & 1, p.err, ERR_ATTN_TIMEOUT)) {
            ok = false;
            break;
          }
          tc_fence_after();
          issue_pv(1, j);
          if (next) issue_s(1, j + 1);
        }
        umma_commit(&v_empty[vst]);
        if (next) umma_commit(&k_empty[(j + 1) % KS]);
      }
    }
  } else {
    // ---------------- softmax warpgroups: two threads per query row r of tile i
    const int i = (warp - 2) >> 3;          // query tile
    const int hk = ((warp - 2) >> 2) & 1;   // key half of the 128-key tile: [64*hk, 64*hk+64)
    const int q = warp & 3;                 // TMEM lane quadrant
    const int r = q * 32 + lane;
    const int bar_id = 1 + i;               // named barrier of this tile's 8 warps
    const bool active = (i == 0 || has_q1);
    const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
    const uint32_t s_addr = tmem + i * KT + lane_off;
    const uint32_t o_addr = tmem + 2 * KT + i * 128 + lane_off + hk * (DH / 2);
    float* xch = reinterpret_cast<float*>(tmem_slot + 4) + i * 2 * QT;  // [2 halves][128 rows]
    float m = -INFINITY, l = 0.0f;  // l: this thread's half of the row sum
    bool ok = true;
    constexpr int KH = KT / 2;      // keys per thread
    if (active) {
      const float sl2 = p.scale_log2;
      // Every warp of the tile runs all nT iterations and every named barrier,
      // also after a failed wait (which only skips the work), so the barrier
      // counts always match.
      for (int j = 0; j < nT; ++j) {
        if (ok) ok = warp_wait(&s_full[i], j & 1, p.err);
        const int key0 = (j_begin + j) * KT + hk * KH;
        const bool ragged = key0 + KH > kv_len;
        float mx_half = -INFINITY;
        if (ok) {
          // pass 1: row max of this thread's 64 keys, 32 columns at a time
          tc_fence_after();
#pragma unroll
          for (int c = 0; c < KH / 32; ++c) {
            float s[32];
            tmem_ld32(s_addr + hk * KH + c * 32, s);
            tmem_wait_ld();
            if (ragged) {
#pragma unroll
              for (int e = 0; e < 32; ++e)
                if (key0 + c * 32 + e >= kv_len) s[e] = -INFINITY;
            }
            float m4[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) m4[e] = max3(s[e], s[e + 4], s[e + 8]);
#pragma unroll
            for (int e = 0; e < 4; ++e) m4[e] = max3(m4[e], s[e + 12], s[e + 16]);
#pragma unroll
            for (int e = 0; e < 4; ++e) m4[e] = max3(m4[e], s[e + 20], s[e + 24]);
#pragma unroll
            for (int e = 0; e < 4; ++e) m4[e] = fmaxf(m4[e], s[e + 28]);
            mx_half = max3(mx_half, fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
          }
        }
        // Row max over both key halves (shared-memory exchange).
        xch[hk * QT + r] = mx_half;
        asm volatile("bar.sync %0, 256;" ::"r"(bar_id) : "memory");
        const float other_mx = xch[(1 - hk) * QT + r];
        asm volatile("bar.sync %0, 256;" ::"r"(bar_id) : "memory");
        if (!ok) continue;
        const float m_tile = fmaxf(mx_half, other_mx) * sl2;
        const bool grow = m_tile > m + kRescaleThreshold;
        if (__any_sync(0xffffffffu, grow)) {
          const float m_new = grow ? m_tile : m;
          const float alpha = grow ? fast_exp2(m - m_new) : 1.0f;
          if (j > 0) {
            // PV_{i,j-1} completed before S_{i,j} (in-order MMAs): O_i is stable.
#pragma unroll 1
            for (int c = 0; c < Cfg::OH / Cfg::OC; ++c) {
              float o[Cfg::OC];
              o_ld<Cfg::OC>(o_addr + c * Cfg::OC, o);
              tmem_wait_ld();
#pragma unroll
              for (int e = 0; e < Cfg::OC; ++e) o[e] *= alpha;
              o_st<Cfg::OC>(o_addr + c * Cfg::OC, o);
            }
          }
          l *= alpha;
          m = m_new;
        }
        // pass 2: P = exp2(s * scale_log2 - m) in bf16.  Chunk c of this
        // thread's keys goes to packed columns [64 hk + 16 c, +16), which only
        // overlap S columns this thread has already consumed.
        const float negm = -m;
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int c = 0; c < KH / 32; ++c) {
          float s[32];
          tmem_ld32(s_addr + hk * KH + c * 32, s);
          tmem_wait_ld();
          if (ragged) {
#pragma unroll
            for (int e = 0; e < 32; ++e)
              if (key0 + c * 32 + e >= kv_len) s[e] = -INFINITY;
          }
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            float a = s[2 * e], b = s[2 * e + 1];
            ffma2(a, b, sl2, negm);
            a = fast_exp2(a);
            b = fast_exp2(b);
            fadd2(acc[2 * (e & 1)], acc[2 * (e & 1) + 1], a, b);
            pk[e] = pack_bf16x2(a, b);
          }
          tmem_st16(s_addr + hk * KH + c * 16, pk);
        }
        tmem_wait_st();
        l += (acc[0] + acc[1]) + (acc[2] + acc[3]);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_full[i]);
      }
      if (ok) ok = warp_wait(&o_done[i], (nT - 1) & 1, p.err);
      if (ok) tc_fence_after();
      // Row sum over both key halves, fixed order (half 0 + half 1).
      xch[hk * QT + r] = l;
      asm volatile("bar.sync %0, 256;" ::"r"(bar_id) : "memory");
      l = xch[r] + xch[QT + r];
    }
    const bool valid = active && (pair * 2 * QT + i * QT + r) < p.T;
    __nv_bfloat16* dst =
        p.o + static_cast<int64_t>(qrow0 + i * QT + r) * p.d + head * DH + hk * (DH / 2);
    auto store_row = [&](const float* o, int c, float inv) {
      uint4* d4 = reinterpret_cast<uint4*>(dst + c * Cfg::OC);
#pragma unroll
      for (int e = 0; e < Cfg::OC / 8; ++e) {
        uint4 w;
        w.x = pack_bf16x2(o[8 * e + 0] * inv, o[8 * e + 1] * inv);
        w.y = pack_bf16x2(o[8 * e + 2] * inv, o[8 * e + 3] * inv);
        w.z = pack_bf16x2(o[8 * e + 4] * inv, o[8 * e + 5] * inv);
        w.w = pack_bf16x2(o[8 * e + 6] * inv, o[8 * e + 7] * inv);
        d4[e] = w;
      }
    };
    if (nsplit == 1) {
      if (active && ok) {
        const float inv_l = 1.0f / l;
#pragma unroll 1
        for (int c = 0; c < Cfg::OH / Cfg::OC; ++c) {
          float o[Cfg::OC];
          o_ld<Cfg::OC>(o_addr + c * Cfg::OC, o);
          tmem_wait_ld();
          if (valid) store_row(o, c, inv_l);
        }
      }
    } else {
      // Leave this key-half CTA's unnormalised O, m, l; the second CTA of the
      // query pair to arrive merges both.
      constexpr int PART = (DH + 2) * QT;
      float* base = p.part + static_cast<int64_t>(item) * 4 * PART;
      float* mine = base + (half * 2 + i) * PART;
      const float* other = base + ((1 - half) * 2 + i) * PART;
      if (active && ok) {
#pragma unroll 1
        for (int c = 0; c < Cfg::OH / Cfg::OC; ++c) {
          float o[Cfg::OC];
          o_ld<Cfg::OC>(o_addr + c * Cfg::OC, o);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < Cfg::OC; ++e) mine[(hk * Cfg::OH + c * Cfg::OC + e) * QT + r] = o[e];
        }
        if (hk == 0) {
          mine[DH * QT + r] = m;
          mine[(DH + 1) * QT + r] = l;
        }
      }
      __threadfence();
      asm volatile("bar.sync 3, 512;" ::: "memory");
      if (warp == 2 && lane == 0)
        *s_last_p = (ok && !error_raised(p.err)) ? atomicAdd(&p.counters[item], 1) : -1;
      asm volatile("bar.sync 3, 512;" ::: "memory");
      if (*s_last_p == 1) {
        __threadfence();
        if (active) {
          const float* h0 = half == 0 ? mine : other;
          const float* h1 = half == 0 ? other : mine;
          const float m0 = __ldcg(h0 + DH * QT + r), m1 = __ldcg(h1 + DH * QT + r);
          const float l0 = __ldcg(h0 + (DH + 1) * QT + r), l1 = __ldcg(h1 + (DH + 1) * QT + r);
          const float mm = fmaxf(m0, m1);
          const float a0 = fast_exp2(m0 - mm), a1 = fast_exp2(m1 - mm);
          const float inv = 1.0f / (l0 * a0 + l1 * a1);
#pragma unroll 1
          for (int c = 0; c < Cfg::OH / Cfg::OC; ++c) {
            float o[Cfg::OC];
#pragma unroll
            for (int e = 0; e < Cfg::OC; ++e) {
              const int k = (hk * Cfg::OH + c * Cfg::OC + e) * QT + r;
              o[e] = __ldcg(h0 + k) * a0 + __ldcg(h1 + k) * a1;
            }
            if (valid) store_row(o, c, inv);
          }
        }
        if (warp == 2 && lane == 0) p.counters[item] = 0;
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
                      const AttnParams& p, int n_tasks, int grid, cudaStream_t st) {
  static bool attr_set = false;
  const size_t smem = attn_smem_bytes(DH);
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel<DH>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  AttnParams q = p;
  q.n_tasks = n_tasks;
  attn_tc_kernel<DH><<<grid, kThreads, smem, st>>>(*tmQ, *tmK, *tmV, q);
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
  // Every variant asks for more than half the SM's shared memory so that one
  // CTA holds an SM: the 512 TMEM columns it allocates are then always free.
  const size_t one_per_sm = 120 * 1024;
  static_assert(AttnCfg<128>::SMEM <= 232448, "attention shared memory over the per-block limit");
  return need > one_per_sm ? need : one_per_sm;
}

cudaError_t launch_attention(const CUtensorMap* tmQ, const CUtensorMap* tmK,
                             const CUtensorMap* tmV, const AttnParams& p, int n_tasks, int grid,
                             cudaStream_t st) {
  if (grid <= 0) return cudaSuccess;
  switch (p.dh) {
    case 32: return launch_dh<32>(tmQ, tmK, tmV, p, n_tasks, grid, st);
    case 64: return launch_dh<64>(tmQ, tmK, tmV, p, n_tasks, grid, st);
    case 128: return launch_dh<128>(tmQ, tmK, tmV, p, n_tasks, grid, st);
    default: return cudaErrorInvalidValue;
  }
}

namespace {
__global__ void fill_attn_tasks_kernel(TaskDev* tasks, int n, int T, int L) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  TaskDev t{};
  t.row0 = i * T;
  t.ring0 = i;
  t.kv_len = L;
  tasks[i] = t;
}
}  // namespace

cudaError_t launch_fill_attn_tasks(TaskDev* tasks, int n, int T, int L, cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  fill_attn_tasks_kernel<<<(n + 127) / 128, 128, 0, st>>>(tasks, n, T, L);
  return cudaGetLastError();
}

int attn_grid_size(const int* kv_lens, int n_tasks, int T, int H) {
  const int n_pairs = (T + 2 * QT - 1) / (2 * QT);
  int total = 0;
  for (int t = 0; t < n_tasks; ++t) {
    const int ns = ((kv_lens[t] + KT - 1) / KT >= kAttnSplitMinTiles) ? 2 : 1;
    total += H * n_pairs * ns;
  }
  return total;
}

size_t attn_part_floats(int max_tasks, int T, int H, int dh) {
  const int n_pairs = (T + 2 * QT - 1) / (2 * QT);
  return static_cast<size_t>(max_tasks) * H * n_pairs * 4 * (dh + 2) * QT;
}

}  // namespace psv
