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
// CTA pairs (clusters of two SMs) with 2-SM tcgen05 MMAs (cta_group::2).  A
// work piece is 256 query rows of one (task, head), 128 per CTA, over the
// whole window or one fixed half of it, walked in tiles of 256 keys.  Per key
// tile j the even CTA issues
//   S_j  = Q K_j^T     M=256, N=256, K=dh    (each CTA holds 128 of the keys)
//   O   += P_j V_j     M=256, N=dh,  K=256   (each CTA holds dh/2 rows of V^T)
// S, P (bf16, two per TMEM column) and O have TMEM columns of their own, so
// S_{j+1} runs while the softmax works on S_j, and P_{j-1}.V_{j-1} runs while
// it computes the exponentials of tile j.  The wide S MMA (N=256) keeps the one
// issuing thread well ahead of the tensor pipe.  Warp roles, 384 threads in
// three warpgroups:
//   warp 0       TMA: per piece the Q tile, then this CTA's K halves (3 stages);
//                on the even CTA also the reader of the work queue
//   warp 1       TMEM allocator (both CTAs) and MMA issuer (even CTA)
//   warp 2       TMA: this CTA's V^T halves (3 stages)
//   warps 4..11  softmax, two threads per query row in one warp (lanes l
//                and l + 16), 128 keys each of a 256-key tile, through
//                16-lane TMEM accesses: the row max and sum need one
//                shuffle, no shared memory and no barrier; online max/sum in
//                the log2 domain with lazy O rescale (only when the running
//                max grows by more than 2^8)
// The first warpgroup hands registers to the two softmax warpgroups
// (setmaxnreg), so that a softmax thread holds its 128 scores without
// spilling: local-memory traffic would compete with the MMAs' shared-memory
// operand reads.
// Persistent pairs (at most one per two SMs) take pieces from a work queue (a
// device counter, rewound by the last pair to finish) in a fixed order, large
// pieces first: the loads, MMAs and softmax run on across piece boundaries
// (barrier phases and stages count tiles over all of a pair's pieces), so the
// next piece's Q load and first S MMA overlap the previous piece's last tile
// and epilogue, and a pair that finishes early takes more work instead of
// leaving its SMs idle for the rest of the launch.
// Long windows (>= kAttnSplitMinTiles key tiles) and the short tail units
// (whose rows fit in the even CTA) are split into two fixed key halves; each
// half leaves its unnormalised O, m and l in a partial area and the CTA that
// arrives second on its counter merges both in a fixed order (half 0, half 1).
// The split depends only on the task's window length and the unit, and the
// merge order is fixed, so a task's result depends neither on which pair took
// which piece nor on the rest of the wave.
#include "psv_device.cuh"
#include "psv_kernels.h"

namespace psv {

namespace {

constexpr int QT = 128;   // query rows per CTA (256 per pair)
constexpr int KT = 256;   // keys per tile
constexpr uint32_t TMEM_COLS = 512;
constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr int kThreads = 384;
constexpr int kStages = 3;                 // K and V^T stages
// Register split: the first warpgroup shrinks to kRegsLow per thread, the two
// softmax warpgroups grow to kRegsHigh.  The block's launch allocation
// (threads x registers at launch) must cover the split; the host checks it
// before the first launch (kRegsNeeded).
constexpr int kRegsLow = 64, kRegsHigh = 216;
constexpr int kRegsNeeded = 128 * kRegsLow + 256 * kRegsHigh;
// Tails of head h are queued after the non-tail pieces of head h + kTailDelay
// of the same task (see decode_piece).
constexpr int kTailDelay = 4;
// Threads of a pair that take each work piece: the even CTA's MMA issuer, and
// in both CTAs the V^T loader and one softmax thread; the odd CTA's Q/K loader
// (the even CTA's one publishes the pieces).
constexpr int kPieceReaders = 6;

template <int DH>
struct AttnCfg {
  static constexpr int AW = DH < 64 ? DH : 64;  // elements per swizzle row (Q, K)
  static constexpr int ROWB = AW * 2;           // bytes per swizzle row
  static constexpr int NA = DH / AW;            // atoms along dh
  static constexpr int VR = DH / 2;             // V^T rows held per CTA
  static constexpr int Q_BYTES = QT * DH * 2;
  static constexpr int K_BYTES = 128 * DH * 2;  // this CTA's 128 keys of a tile
  static constexpr int V_BYTES = VR * KT * 2;   // this CTA's dh/2 rows x 256 keys
  static constexpr int Q_ATOM = QT * ROWB;
  static constexpr int K_ATOM = 128 * ROWB;
  static constexpr int V_ATOM = VR * 128;       // [dh/2 rows][64 keys]
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + Q_BYTES;
  static constexpr int OFF_V = OFF_K + kStages * K_BYTES;
  static constexpr int OFF_BAR = OFF_V + kStages * V_BYTES;
  static constexpr int N_BARS = 12 + 4 * kStages;
  // barriers, the TMEM address word and the merge flag, two published piece
  // slots and the softmax warps' copy (two int4 each: the piece and its task
  // fields).  The dynamic shared-memory window starts 1024-byte aligned (no
  // static shared variables; checked at run time).
  static constexpr size_t SMEM = OFF_BAR + N_BARS * 8 + 16 + 6 * 16;
  static constexpr int OH = DH / 2;              // O columns per thread
  static constexpr int OC = OH < 32 ? OH : 32;   // O columns per TMEM access
  static_assert(V_ATOM % 1024 == 0 && K_ATOM % 1024 == 0, "swizzle atoms stay 1024-aligned");
};

// TMEM columns of each CTA: S [0, 256), P [256, 384), O [384, 384 + dh).
constexpr uint32_t COL_S = 0, COL_P = 256, COL_O = 384;

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, int* err) {
  int ok = 0;
  if (lane_id() == 0) ok = mbar_wait(bar, parity, err, ERR_ATTN_TIMEOUT) ? 1 : 0;
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// 2-SM MMA with A from TMEM (P: each CTA's 128 rows in its own TMEM) and B
// from shared memory (each CTA's N/2 rows of V^T at the same offset).
__device__ __forceinline__ void umma_pair_tmem_a(uint32_t tmem_d, uint32_t tmem_a, uint64_t bdesc,
                                                 uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(tmem_d),
      "r"(tmem_a), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// 16-lane accesses of TMEM (shape 16x32bx2): threads 0-15 of the warp reach
// lanes [base, base + 16) at column c, threads 16-31 the same lanes at column
// c + SPLIT.  This lets the two threads of a query row that hold the two
// halves of its keys (or of its O columns) sit in one warp, so the row's max
// and sum are combined with one shuffle.
template <int SPLIT>
__device__ __forceinline__ void tmem_ld16x2_32(uint32_t taddr, float* v) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.16x32bx2.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32], %33;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr), "n"(SPLIT));
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

template <int SPLIT>
__device__ __forceinline__ void tmem_ld16x2_16(uint32_t taddr, float* v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.16x32bx2.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16], %17;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr), "n"(SPLIT));
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

template <int SPLIT>
__device__ __forceinline__ void tmem_st16x2_16(uint32_t taddr, const uint32_t* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.16x32bx2.x16.b32 [%0], %1, "
      "{%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17};" ::"r"(taddr),
      "n"(SPLIT), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]),
      "r"(v[7]), "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]),
      "r"(v[14]), "r"(v[15])
      : "memory");
}

template <int SPLIT>
__device__ __forceinline__ void tmem_st16x2_32f(uint32_t taddr, const float* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.16x32bx2.x32.b32 [%0], %1, "
      "{%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,"
      "%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33};" ::"r"(taddr),
      "n"(SPLIT), "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])),
      "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])),
      "r"(__float_as_uint(v[5])), "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])),
      "r"(__float_as_uint(v[8])), "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])),
      "r"(__float_as_uint(v[11])), "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])),
      "r"(__float_as_uint(v[14])), "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])),
      "r"(__float_as_uint(v[17])), "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])),
      "r"(__float_as_uint(v[20])), "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])),
      "r"(__float_as_uint(v[23])), "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])),
      "r"(__float_as_uint(v[26])), "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])),
      "r"(__float_as_uint(v[29])), "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
      : "memory");
}

// O-column access of OC (16 or 32) f32 columns of this thread's half of its
// row's O: columns [c, c + OC) for threads 0-15, [c + OH, c + OH + OC) for
// threads 16-31.
template <int OC, int OH>
__device__ __forceinline__ void o_ld(uint32_t taddr, float* v) {
  if constexpr (OC == 32) tmem_ld16x2_32<OH>(taddr, v);
  else tmem_ld16x2_16<OH>(taddr, v);
}
template <int OH>
__device__ __forceinline__ void o_st16(uint32_t taddr, const float* v) {
  uint32_t u[16];
#pragma unroll
  for (int e = 0; e < 16; ++e) u[e] = __float_as_uint(v[e]);
  tmem_st16x2_16<OH>(taddr, u);
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

// At least one tile per piece (every piece runs the same barrier sequence).
__host__ __device__ __forceinline__ int n_key_tiles(int kv_len) {
  return kv_len > KT ? (kv_len + KT - 1) / KT : 1;
}
__host__ __device__ __forceinline__ int n_units_of(int T) { return (T + 2 * QT - 1) / (2 * QT); }
// The last query unit of a task is a tail when all its rows sit in the even
// CTA (T = 1560: 24 rows).  A tail costs a full unit's MMAs and softmax.
__host__ __device__ __forceinline__ bool has_tail(int T) {
  return T - (n_units_of(T) - 1) * 2 * QT <= QT;
}
// Key halves of a (task, head, query unit): a function of the task's window
// and of the unit being a tail only, never of the rest of the launch.  Long
// windows are split for parallelism; tails are split so that their short
// halves fill the end of the launch.
__host__ __device__ __forceinline__ int n_splits(int kv_len, bool tail) {
  const int nt = n_key_tiles(kv_len);
  if (nt >= kAttnSplitMinTiles) return 2;
  if (tail && nt >= kAttnTailSplitMinTiles) return 2;
  return 1;
}
__host__ __device__ __forceinline__ int pieces_main(int kv_len, int T, int H) {
  return H * (n_units_of(T) - (has_tail(T) ? 1 : 0)) * n_splits(kv_len, false);
}
__host__ __device__ __forceinline__ int pieces_tail(int kv_len, int T, int H) {
  return has_tail(T) ? H * n_splits(kv_len, true) : 0;
}

// Work piece k of the queue -> {task, head, query unit, half | halves << 8};
// x = -1 past the end.  Order, task by task: the non-tail pieces of one
// (task, head) together (the pairs that share its K/V window run at the same
// time), and the tail pieces of head h after the non-tail pieces of head
// h + kTailDelay, while head h's window is still in L2 — except for the last
// F (task, head) groups of the launch, F = a quarter of the pairs, whose tails
// close the queue: short pieces that even out the end of the launch, and few
// enough that the windows of those last groups are still in L2 when their
// tails run.  (All tails at the end made the tail phase of an 8-stream wave
// DRAM-bound: every tail half re-read its window; interleaving all of them
// left long pieces at the end; with F = half the pairs the final tails
// re-read ~120 MB of a 1.3B-shaped launch's 211 MB of Q, K and V.)
__device__ int4 decode_piece(int k, const AttnParams& p) {
  if (k < 0 || k >= p.n_pieces) return make_int4(-1, 0, 0, 0);
  const int nu = n_units_of(p.T);
  const bool tail = has_tail(p.T);
  const int nm = nu - (tail ? 1 : 0);
  const int G = p.n_tasks * p.H;
  const int pairs = static_cast<int>(gridDim.x / 2);
  const int F = tail ? min(G, (pairs + 3) / 4) : 0;  // groups whose tails close the queue
  const int gf = G - F;
  const int D = min(kTailDelay, p.H);
  for (int t = 0; t < p.n_tasks; ++t) {
    const int kv = p.tasks[t].kv_len;
    const int nsm = n_splits(kv, false), nst = tail ? n_splits(kv, true) : 0;
    const int a = nm * nsm, b = nst;  // pieces of one head: non-tail, tail
    const int hf = min(max(gf - t * p.H, 0), p.H);  // heads [0, hf) interleave their tails
    const int hb = min(hf, p.H - D);                 // ... after the head D further on
    const int c = p.H * a + hf * b;
    if (k >= c) {
      k -= c;
      continue;
    }
    auto main_piece = [&](int h, int i) { return make_int4(t, h, i / nsm, (i % nsm) | (nsm << 8)); };
    auto tail_piece = [&](int h, int i) { return make_int4(t, h, nu - 1, i | (nst << 8)); };
    if (k < D * a) return main_piece(k / a, k % a);
    k -= D * a;
    if (k < hb * (a + b)) {
      const int blk = k / (a + b), off = k % (a + b);
      return off < a ? main_piece(D + blk, off) : tail_piece(blk, off - a);
    }
    k -= hb * (a + b);
    if (k < (p.H - D - hb) * a) return main_piece(D + hb + k / a, k % a);
    k -= (p.H - D - hb) * a;
    if (b == 0) break;
    return tail_piece(hb + k / b, k % b);
  }
  if (tail) {
    for (int t = 0; t < p.n_tasks; ++t) {
      const int nst = n_splits(p.tasks[t].kv_len, true);
      const int hf = min(max(gf - t * p.H, 0), p.H);
      const int c = (p.H - hf) * nst;
      if (k < c) return make_int4(t, hf + k / nst, nu - 1, (k % nst) | (nst << 8));
      k -= c;
    }
  }
  return make_int4(-1, 0, 0, 0);
}

struct Piece {
  int ti, head, unit, half, nsplit;
  int j_begin, nT;  // key tiles [j_begin, j_begin + nT) of the window
  int kv_len, row0, ring;
};

// The task fields a piece needs, published with it: {kv_len, row0, ring}.
__device__ __forceinline__ int4 piece_task(int4 pc, const AttnParams& p) {
  if (pc.x < 0) return make_int4(0, 0, 0, 0);
  const TaskDev& task = p.tasks[pc.x];
  return make_int4(task.kv_len, task.row0, task.ring0 + p.block * p.S, 0);
}

__device__ __forceinline__ Piece piece_of(int4 pc, int4 pt) {
  Piece g;
  g.ti = pc.x;
  g.head = pc.y;
  g.unit = pc.z;
  g.half = pc.w & 0xff;
  g.nsplit = pc.w >> 8;
  g.kv_len = pt.x;
  g.row0 = pt.y;
  g.ring = pt.z;
  const int nt = n_key_tiles(g.kv_len);
  g.j_begin = g.half == 0 ? 0 : nt / 2;
  g.nT = ((g.nsplit == 1 || g.half == 1) ? nt : nt / 2) - g.j_begin;
  return g;
}

// The piece slots are written by the even CTA's thread with st.shared::cluster
// and published with a release.cluster arrive; readers in either CTA wait
// with an acquire at cluster scope.
__device__ __forceinline__ void st_cluster_v4(uint32_t addr, int4 v) {
  asm volatile("st.shared::cluster.v4.s32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}

// One 32-byte global store (a whole sector); ptr 32-byte aligned.
__device__ __forceinline__ void st_global_v8(void* ptr, const uint32_t* w) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(ptr), "r"(w[0]),
               "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
               : "memory");
}

__device__ __forceinline__ int4 ld_shared_v4(const void* ptr) {
  int4 v;
  asm volatile("ld.shared.v4.s32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(smem_u32(ptr))
               : "memory");
  return v;
}

__device__ __forceinline__ bool mbar_try_wait_acq_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// mbar_wait with cluster-scope acquire (bounded the same way).
__device__ __forceinline__ bool mbar_wait_acq_cluster(uint64_t* bar, uint32_t parity, int* err,
                                                      int code) {
  if (mbar_try_wait_acq_cluster(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t i = 0;; ++i) {
    if (mbar_try_wait_acq_cluster(bar, parity)) return true;
    if ((i & 63) == 63) {
      if (error_raised(err)) return false;
      if (global_timer_ns() - t0 > kWaitLimitNs) {
        raise_error(err, code);
        return false;
      }
    }
  }
}

template <int DH>
__global__ void __launch_bounds__(kThreads, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tmQ,
                   const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const AttnParams p) {
  using Cfg = AttnCfg<DH>;
  constexpr int KS = kStages, VS = kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw;
  // Swizzled TMA tiles need 1024-byte alignment.  The offset of the dynamic
  // window is the same in both CTAs of the pair, so both leave here together.
  if (smem_u32(smem) & 1023) {
    if (threadIdx.x == 0) raise_error(p.err, ERR_BOUNDS);
    return;
  }
  uint8_t* sQ = smem + Cfg::OFF_Q;
  uint8_t* sK = smem + Cfg::OFF_K;
  uint8_t* sV = smem + Cfg::OFF_V;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Cfg::OFF_BAR);
  uint64_t* q_full = bars + 0;        // even CTA: both Q tiles of the current piece landed
  uint64_t* s_full = bars + 1;        // both CTAs: S of a tile in TMEM
  uint64_t* s_free = bars + 2;        // even CTA: all 16 softmax warps of the pair read S
  uint64_t* p_full_a = bars + 3;      // even CTA: all 16 softmax warps wrote the first half of P
  uint64_t* o_done = bars + 4;        // both CTAs: P.V of a tile done (P consumed, O stable)
  uint64_t* p_full_b = bars + 5;      // even CTA: ... and the second half
  uint64_t* q_empty = bars + 6;       // both CTAs: the last S MMA of a piece is done
  uint64_t* pc_full = bars + 8;       // [2] both CTAs: piece slot published
  uint64_t* pc_empty = bars + 10;     // [2] even CTA: the pair's six readers took the slot
  uint64_t* k_full = bars + 12;       // [KS] even CTA: both K halves of a stage landed
  uint64_t* k_empty = k_full + KS;    // [KS] both CTAs: the S MMA of a stage is done
  uint64_t* v_full = k_empty + KS;    // [VS] even CTA
  uint64_t* v_empty = v_full + VS;    // [VS] both CTAs
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + Cfg::N_BARS);
  int* s_last_p = reinterpret_cast<int*>(tmem_slot + 1);
  int4* pc_slot = reinterpret_cast<int4*>(tmem_slot + 4);   // [2][2] published pieces
  int4* sm_piece = pc_slot + 4;                             // [2] the softmax warps' copy

  pdl_trigger();
  const int warp = warp_id(), lane = lane_id();
  const int rank = static_cast<int>(cluster_ctarank());
  const bool leader = rank == 0;
  if (warp == 0 && lane == 0) {
    for (int i = 0; i < Cfg::N_BARS; ++i) {
      // s_free, p_full_a, p_full_b: every softmax warp of both CTAs arrives
      const bool all16 = i == 2 || i == 3 || i == 5;
      const bool readers = i == 10 || i == 11;
      mbar_init(&bars[i], all16 ? 16 : (readers ? kPieceReaders : 1));
    }
    fence_mbar_init();
    prefetch_tensormap(&tmQ);
    prefetch_tensormap(&tmK);
    prefetch_tensormap(&tmV);
  }
  if (warp == 1) tmem_alloc_pair(tmem_slot, TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  // The peer's barriers must be initialised before anything signals them.
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // Everything above overlaps the previous kernel's tail; from here on the
  // kernel reads what earlier kernels wrote (task table, work queue).
  pdl_wait();
  const uint32_t pc_empty0 = mapa_shared(pc_empty, 0);
  // A reader of the pair takes piece i from slot i & 1 and acknowledges it on
  // the even CTA (after it has used the values, so the slot may be reused).
  auto take_piece = [&](int i, int4& pc, int4& pt) -> bool {
    if (!mbar_wait_acq_cluster(&pc_full[i & 1], (i >> 1) & 1, p.err, ERR_ATTN_TIMEOUT)) return false;
    pc = ld_shared_v4(&pc_slot[2 * (i & 1)]);
    pt = ld_shared_v4(&pc_slot[2 * (i & 1) + 1]);
    mbar_arrive_remote(pc_empty0 + (i & 1) * 8);
    return true;
  };

  if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsLow));
    if (warp == 0) {
      if (lane == 0) {
        // ---------------- TMA: per piece the Q tile, then this CTA's K halves
        // (3 stages, counted over all pieces); completion on the even CTA.
        // The even CTA's thread also takes the pieces from the work queue and
        // publishes them to both CTAs.
        const uint32_t q_full0 = mapa_shared(q_full, 0);
        const uint32_t k_full0 = mapa_shared(k_full, 0);
        int gk = 0;
        for (int i = 0;; ++i) {
          int4 pc, pt;
          if (leader) {
            const int b = i & 1;
            if (i >= 2 && !mbar_wait(&pc_empty[b], ((i >> 1) - 1) & 1, p.err, ERR_ATTN_TIMEOUT)) break;
            pc = decode_piece(atomicAdd(p.counters, 1), p);
            pt = piece_task(pc, p);
            for (uint32_t r = 0; r < 2; ++r) {
              st_cluster_v4(mapa_shared(&pc_slot[2 * b], r), pc);
              st_cluster_v4(mapa_shared(&pc_slot[2 * b + 1], r), pt);
            }
            for (uint32_t r = 0; r < 2; ++r) mbar_arrive_cluster(mapa_shared(&pc_full[b], r));
          } else if (!take_piece(i, pc, pt)) {
            break;
          }
          if (pc.x < 0) break;
          const Piece pg = piece_of(pc, pt);
          // The Q buffer is reused once the previous piece's S MMAs are done.
          if (i > 0 && !mbar_wait(q_empty, (i - 1) & 1, p.err, ERR_ATTN_TIMEOUT)) break;
          if (leader) mbar_arrive_expect_tx(q_full, 2 * Cfg::Q_BYTES);
#pragma unroll
          for (int a = 0; a < Cfg::NA; ++a)
            tma_load_2d_pair(sQ + a * Cfg::Q_ATOM, &tmQ, q_full0, pg.head * DH + a * Cfg::AW,
                             pg.row0 + pg.unit * 2 * QT + rank * QT);
          bool ok = true;
          for (int j = 0; j < pg.nT; ++j, ++gk) {
            const int st = gk % KS;
            if (!mbar_wait(&k_empty[st], ((gk / KS) & 1) ^ 1, p.err, ERR_ATTN_TIMEOUT)) {
              ok = false;
              break;
            }
            if (leader) mbar_arrive_expect_tx(&k_full[st], 2 * Cfg::K_BYTES);
            uint8_t* dst = sK + st * Cfg::K_BYTES;
#pragma unroll
            for (int a = 0; a < Cfg::NA; ++a)
              tma_load_3d_pair(dst + a * Cfg::K_ATOM, &tmK, k_full0 + st * 8, pg.head * DH + a * Cfg::AW,
                               (pg.j_begin + j) * KT + rank * 128, pg.ring);
          }
          if (!ok) break;
        }
        // Stay until the MMAs released the last stages (bounded): no copy into
        // or read of this CTA's shared memory may be left when it exits.
        const uint64_t t0 = global_timer_ns();
        for (int j = (gk > KS ? gk - KS : 0); j < gk; ++j) {
          while (!mbar_try_wait(&k_empty[j % KS], (j / KS) & 1) &&
                 global_timer_ns() - t0 < kWaitLimitNs) {
          }
        }
      }
    } else if (warp == 2) {
      if (lane == 0) {
        // ---------------- TMA: V^T halves (dh/2 rows of this CTA, 256 keys)
        const uint32_t v_full0 = mapa_shared(v_full, 0);
        int gv = 0;
        for (int i = 0;; ++i) {
          int4 pc, pt;
          if (!take_piece(i, pc, pt) || pc.x < 0) break;
          const Piece pg = piece_of(pc, pt);
          bool ok = true;
          for (int j = 0; j < pg.nT; ++j, ++gv) {
            const int st = gv % VS;
            if (!mbar_wait(&v_empty[st], ((gv / VS) & 1) ^ 1, p.err, ERR_ATTN_TIMEOUT)) {
              ok = false;
              break;
            }
            if (leader) mbar_arrive_expect_tx(&v_full[st], 2 * Cfg::V_BYTES);
            uint8_t* dst = sV + st * Cfg::V_BYTES;
#pragma unroll
            for (int a = 0; a < KT / 64; ++a)
              tma_load_3d_pair(dst + a * Cfg::V_ATOM, &tmV, v_full0 + st * 8,
                               (pg.j_begin + j) * KT + a * 64, rank * Cfg::VR, pg.ring * p.H + pg.head);
          }
          if (!ok) break;
        }
        const uint64_t t0 = global_timer_ns();
        for (int j = (gv > VS ? gv - VS : 0); j < gv; ++j) {
          while (!mbar_try_wait(&v_empty[j % VS], (j / VS) & 1) &&
                 global_timer_ns() - t0 < kWaitLimitNs) {
          }
        }
      }
    } else if (warp == 1 && lane == 0 && leader) {
      // ---------------- MMA issuer (even CTA), 2-SM MMAs for the pair.  Per
      // piece: S_0 once its Q is in (and the softmax read the previous tile's
      // S), then per tile j: S_{j+1} once every softmax warp has read S_j (and
      // K_{j+1} is in), P_j.V_j once every softmax warp has written P_j (and
      // V_j is in).  Issue order is execution order; tiles are counted over
      // all pieces of the pair (barrier phases, K/V stages).
      constexpr uint32_t IDESC_S = umma_idesc_bf16(2 * QT, KT);
      constexpr uint32_t IDESC_O = umma_idesc_bf16(2 * QT, DH);
      const uint64_t dq = umma_desc_kmajor(smem_u32(sQ), Cfg::ROWB);
      const uint64_t dk = umma_desc_kmajor(smem_u32(sK), Cfg::ROWB);
      const uint64_t dv = umma_desc_kmajor(smem_u32(sV), 128);
      auto issue_s = [&](int t) {
        const uint64_t b = dk + static_cast<uint64_t>(((t % KS) * Cfg::K_BYTES) >> 4);
#pragma unroll
        for (int kk = 0; kk < DH / 16; ++kk) {
          const int e = kk * 16;
          const uint32_t oq = ((e / Cfg::AW) * Cfg::Q_ATOM + (e % Cfg::AW) * 2) >> 4;
          const uint32_t ok = ((e / Cfg::AW) * Cfg::K_ATOM + (e % Cfg::AW) * 2) >> 4;
          umma_bf16_pair(tmem + COL_S, dq + oq, b + ok, IDESC_S, kk != 0);
        }
        umma_commit_pair_mc(s_full, 0x3);
        umma_commit_pair_mc(&k_empty[t % KS], 0x3);
      };
      int g = 0;  // tiles of earlier pieces
      bool ok = true;
      for (int i = 0; ok; ++i) {
        int4 pc, pt;
        if (!take_piece(i, pc, pt) || pc.x < 0) break;
        const int nT = piece_of(pc, pt).nT;
        if (!mbar_wait(q_full, i & 1, p.err, ERR_ATTN_TIMEOUT) ||
            !mbar_wait(&k_full[g % KS], (g / KS) & 1, p.err, ERR_ATTN_TIMEOUT) ||
            (g > 0 && !mbar_wait(s_free, (g - 1) & 1, p.err, ERR_ATTN_TIMEOUT)))
          break;
        tc_fence_after();
        issue_s(g);
        // After the piece's last S MMA the Q buffer may be refilled once it is done.
        if (nT == 1) umma_commit_pair_mc(q_empty, 0x3);
        for (int j = 0; j < nT; ++j) {
          const int t = g + j;
          if (j + 1 < nT) {
            if (!mbar_wait(s_free, t & 1, p.err, ERR_ATTN_TIMEOUT) ||
                !mbar_wait(&k_full[(t + 1) % KS], ((t + 1) / KS) & 1, p.err, ERR_ATTN_TIMEOUT)) {
              ok = false;
              break;
            }
            tc_fence_after();
            issue_s(t + 1);
            if (j + 2 == nT) umma_commit_pair_mc(q_empty, 0x3);
          }
          // P_j arrives in two halves: keys [0,64) and [128,192) first (the
          // first two chunks of each softmax thread), then the rest, so half
          // of the P.V MMAs issue while the softmax still computes the other
          // half.  A piece's first P.V overwrites O: the softmax warps read
          // the previous piece's O before they wrote any of this P.
          if (!mbar_wait(p_full_a, t & 1, p.err, ERR_ATTN_TIMEOUT) ||
              !mbar_wait(&v_full[t % VS], (t / VS) & 1, p.err, ERR_ATTN_TIMEOUT)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t b = dv + static_cast<uint64_t>(((t % VS) * Cfg::V_BYTES) >> 4);
          auto issue_pv = [&](int kk) {
            // keys [16 kk, 16 kk + 16) of P sit in packed columns [8 kk, 8 kk + 8)
            const uint32_t ov = ((kk >> 2) * Cfg::V_ATOM + (kk & 3) * 32) >> 4;
            umma_pair_tmem_a(tmem + COL_O, tmem + COL_P + kk * 8, b + ov, IDESC_O, (j | kk) != 0);
          };
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) issue_pv(kk);
#pragma unroll
          for (int kk = 8; kk < 12; ++kk) issue_pv(kk);
          if (!mbar_wait(p_full_b, t & 1, p.err, ERR_ATTN_TIMEOUT)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int kk = 4; kk < 8; ++kk) issue_pv(kk);
#pragma unroll
          for (int kk = 12; kk < 16; ++kk) issue_pv(kk);
          umma_commit_pair_mc(o_done, 0x3);
          umma_commit_pair_mc(&v_empty[t % VS], 0x3);
        }
        g += nT;
      }
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsHigh));
    // ---------------- softmax: two threads per query row r of this CTA, in
    // one warp: lanes l and l + 16 hold keys [0, 128) and [128, 256) of a
    // tile of the same row (16-lane TMEM accesses), so the row max and sum
    // are one shuffle away.  Warp 4 + 4h + q serves rows 32 q + 16 h + [0, 16)
    // (q: the TMEM lane quadrant the warp may access).
    const int hk = lane >> 4;         // key half of the tile: keys [128 hk, 128 hk + 128)
    const int q = warp & 3;
    const int rb = q * 32 + ((warp - 4) >> 2) * 16;  // first row of the warp
    const int r = rb + (lane & 15);
    const uint32_t lane_off = static_cast<uint32_t>(rb) << 16;
    const uint32_t s_addr = tmem + COL_S + lane_off;
    const uint32_t p_addr = tmem + COL_P + lane_off;
    const uint32_t o_addr = tmem + COL_O + lane_off;
    const uint32_t s_free0 = mapa_shared(s_free, 0);
    const uint32_t p_full_a0 = mapa_shared(p_full_a, 0);
    const uint32_t p_full_b0 = mapa_shared(p_full_b, 0);
    const float sl2 = p.scale_log2;
    int g = 0;  // tiles of earlier pieces
    for (int i = 0;; ++i) {
      // One thread takes the piece for the CTA's eight softmax warps, so that
      // all of them run the same pieces and named barriers (also after an
      // error, which ends the loop for all).  The copy is rewritten only after
      // every warp has passed this piece's later barriers.
      if (warp == 4 && lane == 0) {
        int4 pc, pt;
        if (!take_piece(i, pc, pt)) pc.x = -1;
        sm_piece[0] = pc;
        sm_piece[1] = pt;
      }
      asm volatile("bar.sync 1, 256;" ::: "memory");
      const int4 pc = ld_shared_v4(sm_piece);
      if (pc.x < 0) break;
      const Piece pg = piece_of(pc, ld_shared_v4(sm_piece + 1));
      const int nT = pg.nT;
      float m = -INFINITY, l = 0.0f;  // l: this thread's half of the row sum
      bool ok = true;
      // Every softmax warp runs all nT iterations and every named barrier, also
      // after a failed wait (which only skips the work), so barrier counts match.
      for (int j = 0; j < nT; ++j) {
        const int t = g + j;
        if (ok) ok = warp_wait(s_full, t & 1, p.err);
        float s[128];
        float mx_half = -INFINITY;
        const int key0 = (pg.j_begin + j) * KT + hk * 128;
        if (ok) {
          tc_fence_after();
#pragma unroll
          for (int c = 0; c < 4; ++c) tmem_ld16x2_32<128>(s_addr + c * 32, s + c * 32);
          tmem_wait_ld();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_remote(s_free0);  // S may now be overwritten
          if (key0 + 128 > pg.kv_len) {
#pragma unroll
            for (int c = 0; c < 128; ++c)
              if (key0 + c >= pg.kv_len) s[c] = -INFINITY;
          }
          float mx8[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) mx8[e] = max3(s[e], s[e + 8], s[e + 16]);
#pragma unroll
          for (int c = 24; c < 120; c += 16) {
#pragma unroll
            for (int e = 0; e < 8; ++e) mx8[e] = max3(mx8[e], s[c + e], s[c + 8 + e]);
          }
#pragma unroll
          for (int e = 0; e < 8; ++e) mx8[e] = fmaxf(mx8[e], s[120 + e]);
          mx_half = fmaxf(max3(mx8[0], mx8[1], mx8[2]),
                          fmaxf(max3(mx8[3], mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
        }
        // Row max over both key halves: the other half is in lane l ^ 16.
        const float other_mx = __shfl_xor_sync(0xffffffffu, mx_half, 16);
        if (!ok) continue;
        const float m_tile = fmaxf(mx_half, other_mx) * sl2;
        const bool grow = m_tile > m + kRescaleThreshold;
        const bool any_grow = __any_sync(0xffffffffu, grow);
        const float m_new = grow ? m_tile : m;
        const float alpha = grow ? fast_exp2(m - m_new) : 1.0f;
        // P = exp2(s * scale_log2 - m) in bf16, 32 keys (16 packed columns) per
        // chunk.  The first two chunks are computed before waiting for the
        // previous tile's P to be consumed, the rest after it.
        const float negm = -m_new;
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        auto exp_chunk = [&](int c, uint32_t* pk) {
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            float a = s[c * 32 + 2 * e], b = s[c * 32 + 2 * e + 1];
            ffma2(a, b, sl2, negm);
            a = fast_exp2(a);
            b = fast_exp2(b);
            fadd2(acc[2 * (e & 3)], acc[2 * (e & 3) + 1], a, b);
            pk[e] = pack_bf16x2(a, b);
          }
        };
        uint32_t pk0[16], pk1[16];
        exp_chunk(0, pk0);
        exp_chunk(1, pk1);
        m = m_new;
        if (j > 0) {
          ok = warp_wait(o_done, (t - 1) & 1, p.err);
          if (!ok) continue;
          tc_fence_after();
        }
        // O is rescaled before the first half of P is released: the P.V MMAs
        // accumulate into it as soon as that half is in.
        if (j > 0 && any_grow) {
#pragma unroll 1
          for (int c = 0; c < Cfg::OH / 16; ++c) {
            float o[16];
            tmem_ld16x2_16<Cfg::OH>(o_addr + c * 16, o);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 16; ++e) o[e] *= alpha;
            o_st16<Cfg::OH>(o_addr + c * 16, o);
          }
        }
        tmem_st16x2_16<64>(p_addr, pk0);
        tmem_st16x2_16<64>(p_addr + 16, pk1);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_remote(p_full_a0);
        exp_chunk(2, pk0);
        tmem_st16x2_16<64>(p_addr + 32, pk0);
        exp_chunk(3, pk1);
        tmem_st16x2_16<64>(p_addr + 48, pk1);
        l = l * alpha + (((acc[0] + acc[1]) + (acc[2] + acc[3])) + ((acc[4] + acc[5]) + (acc[6] + acc[7])));
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_remote(p_full_b0);
      }
      if (ok) ok = warp_wait(o_done, (g + nT - 1) & 1, p.err);
      if (ok) tc_fence_after();
      g += nT;
      // Row sum over both key halves, fixed order (half 0 + half 1).
      {
        const float lo = __shfl_xor_sync(0xffffffffu, l, 16);
        l = hk == 0 ? l + lo : lo + l;
      }
      // O is read (below) before this thread writes any P of the next piece,
      // whose first P.V overwrites it.
      const int qloc0 = pg.unit * 2 * QT + rank * QT;  // first query row of this CTA within the task
      const int item = (pg.ti * p.H + pg.head) * p.max_pairs + pg.unit;
      const bool valid = (qloc0 + r) < p.T;
      __nv_bfloat16* dst = p.o + static_cast<int64_t>(pg.row0 + qloc0 + r) * p.d + pg.head * DH +
                           hk * Cfg::OH;
      // 32-byte stores (whole sectors) where O rows are 32-byte aligned.
      const bool o32 = ((reinterpret_cast<uintptr_t>(p.o) | (static_cast<uintptr_t>(p.d) * 2)) & 31) == 0;
      auto store_row = [&](const float* v, int c, float inv) {
        uint32_t w[Cfg::OC / 2];
#pragma unroll
        for (int e = 0; e < Cfg::OC / 2; ++e) w[e] = pack_bf16x2(v[2 * e] * inv, v[2 * e + 1] * inv);
        if (o32) {
#pragma unroll
          for (int e = 0; e < Cfg::OC / 16; ++e) st_global_v8(dst + c * Cfg::OC + 16 * e, w + 8 * e);
        } else {
          uint4* d4 = reinterpret_cast<uint4*>(dst + c * Cfg::OC);
#pragma unroll
          for (int e = 0; e < Cfg::OC / 8; ++e) d4[e] = make_uint4(w[4 * e], w[4 * e + 1], w[4 * e + 2], w[4 * e + 3]);
        }
      };
      if (pg.nsplit == 1) {
        if (ok) {
          const float inv_l = 1.0f / l;
#pragma unroll 1
          for (int c = 0; c < Cfg::OH / Cfg::OC; ++c) {
            float o[Cfg::OC];
            o_ld<Cfg::OC, Cfg::OH>(o_addr + c * Cfg::OC, o);
            tmem_wait_ld();
            if (valid) store_row(o, c, inv_l);
          }
        }
      } else {
        // Leave this key half's unnormalised O, m, l; the CTA with the same
        // query rows in the other key half's pair that arrives second merges.
        constexpr int PART = (DH + 2) * QT;
        float* base = p.part + static_cast<int64_t>(item) * 4 * PART;
        float* mine = base + (pg.half * 2 + rank) * PART;
        const float* other = base + ((1 - pg.half) * 2 + rank) * PART;
        int* counter = p.counters + kQueueInts + item * 2 + rank;
        if (ok) {
#pragma unroll 1
          for (int c = 0; c < Cfg::OH / Cfg::OC; ++c) {
            float o[Cfg::OC];
            o_ld<Cfg::OC, Cfg::OH>(o_addr + c * Cfg::OC, o);
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
        asm volatile("bar.sync 2, 256;" ::: "memory");
        if (warp == 4 && lane == 0)
          *s_last_p = (ok && !error_raised(p.err)) ? atomicAdd(counter, 1) : -1;
        asm volatile("bar.sync 2, 256;" ::: "memory");
        if (*s_last_p == 1) {
          __threadfence();
          const float* h0 = pg.half == 0 ? mine : other;
          const float* h1 = pg.half == 0 ? other : mine;
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
          if (warp == 4 && lane == 0) *counter = 0;
        }
        // s_last_p is rewritten only after the next piece's first barrier.
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  // Neither CTA leaves (nor frees the pair's TMEM) before both are done:
  // the peer still signals barriers in this CTA's shared memory until then.
  cluster_sync();
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc_pair(tmem, TMEM_COLS);
  }
  if (leader && warp == 0 && lane == 0) {
    // The last pair to finish rewinds the work queue for the next launch
    // (every pair took its final, empty piece before counting itself done).
    __threadfence();
    if (atomicAdd(p.counters + 1, 1) == static_cast<int>(gridDim.x / 2) - 1) {
      atomicExch(p.counters, 0);
      atomicExch(p.counters + 1, 0);
    }
  }
}

template <int DH>
cudaError_t launch_dh(const CUtensorMap* tmQ, const CUtensorMap* tmK, const CUtensorMap* tmV,
                      const AttnParams& p, int grid, cudaStream_t st) {
  static uint64_t set_up = 0;
  const size_t smem = attn_smem_bytes(DH);
  cudaError_t e = once_per_device(&set_up, [&](int) {
    // The register split must fit the launch allocation, else the growing
    // warpgroups would wait for registers forever.
    cudaFuncAttributes fa;
    cudaError_t r = cudaFuncGetAttributes(&fa, attn_tc_kernel<DH>);
    if (r != cudaSuccess) return r;
    if (fa.numRegs * kThreads < kRegsNeeded || fa.numRegs < kRegsLow || fa.numRegs > kRegsHigh)
      return cudaErrorInvalidConfiguration;
    return cudaFuncSetAttribute(attn_tc_kernel<DH>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(smem));
  });
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, attn_tc_kernel<DH>, *tmQ, *tmK, *tmV, p);
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
  if (grid % 2 != 0) return cudaErrorInvalidValue;  // whole CTA pairs only
  AttnParams q = p;
  q.n_tasks = n_tasks;
  switch (p.dh) {
    case 32: return launch_dh<32>(tmQ, tmK, tmV, q, grid, st);
    case 64: return launch_dh<64>(tmQ, tmK, tmV, q, grid, st);
    case 128: return launch_dh<128>(tmQ, tmK, tmV, q, grid, st);
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

int attn_units(int T) { return (T + 2 * QT - 1) / (2 * QT); }

int attn_pieces(const int* kv_lens, int n_tasks, int T, int H) {
  int total = 0;
  for (int t = 0; t < n_tasks; ++t) total += pieces_main(kv_lens[t], T, H) + pieces_tail(kv_lens[t], T, H);
  return total;
}

int attn_pieces_uniform(int L, int n_tasks, int T, int H) {
  return n_tasks * (pieces_main(L, T, H) + pieces_tail(L, T, H));
}

int attn_grid_size(int n_pieces, int sm_count) {
  const int pairs_max = sm_count / 2 > 0 ? sm_count / 2 : 1;
  return 2 * (n_pieces < pairs_max ? n_pieces : pairs_max);
}

size_t attn_part_floats(int max_tasks, int T, int H, int dh) {
  return static_cast<size_t>(max_tasks) * H * attn_units(T) * 4 * (dh + 2) * QT;
}

size_t attn_counter_ints(int max_tasks, int T, int H) {
  return kQueueInts + static_cast<size_t>(max_tasks) * H * attn_units(T) * 2;
}

}  // namespace psv
