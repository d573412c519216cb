// Memory-bound kernels of the wave: adaLN-modulated LayerNorm, the latent
// in-projection, the per-stream conditioning linears, and a dtype cast.
#include "psv_device.cuh"
#include "psv_kernels.h"

namespace psv {

namespace {

constexpr int LN_WARPS = 8;  // rows per CTA (one warp per row)

// Launch with programmatic stream serialization (see pdl_wait).
template <class... KArgs, class... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args... args) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// One warp per row; the row stays in registers (MAXV float4 per lane, d up
// to 128 * MAXV) between the two passes (mean, then centred second moment),
// so h is read once.  The shift/scale vectors of the task of the CTA's first
// row are staged in shared memory by the whole CTA while the rows load, so
// no L2 round trip sits between the statistics and the output; a row of
// another task (only where a task boundary falls inside the CTA's rows)
// reads its vectors from global memory.
template <int MAXV>
__global__ void __launch_bounds__(LN_WARPS * 32)
    ln_mod_kernel(const float* __restrict__ h, __nv_bfloat16* __restrict__ y, int M, int d, int T,
                  const TaskDev* __restrict__ tasks, const float* __restrict__ table,
                  int use_fmod, int block, int shift_off, int scale_off, float eps) {
  extern __shared__ float4 ln_smem[];  // [2][d / 4]: shift, scale
  pdl_trigger();
  pdl_wait();  // h is the previous kernel's output
  const int row0 = blockIdx.x * LN_WARPS;
  const int row = row0 + warp_id();
  const int lane = lane_id();
  const int nv = d >> 2;
  auto mod_base = [&](int r) {
    const TaskDev& t = tasks[r / T];
    return table + (use_fmod ? static_cast<int64_t>(t.fmod0)
                             : static_cast<int64_t>(t.mod0) + static_cast<int64_t>(block) * 6 * d);
  };
  float4 v[MAXV];
  float s = 0.0f;
  if (row < M) {
    const float4* hr = reinterpret_cast<const float4*>(h + static_cast<int64_t>(row) * d);
#pragma unroll
    for (int i = 0; i < MAXV; ++i) {
      const int k = lane + i * 32;
      if (k < nv) {
        v[i] = __ldcs(hr + k);  // read once: keep it out of the way in L2
        s += (v[i].x + v[i].y) + (v[i].z + v[i].w);
      }
    }
  }
  {
    const float* base = mod_base(row0);
    const float4* shift = reinterpret_cast<const float4*>(base + shift_off);
    const float4* scale = reinterpret_cast<const float4*>(base + scale_off);
    for (int k = threadIdx.x; k < nv; k += LN_WARPS * 32) {
      ln_smem[k] = __ldg(shift + k);
      ln_smem[nv + k] = __ldg(scale + k);
    }
  }
  __syncthreads();
  if (row >= M) return;
  const float mean = warp_sum(s) / static_cast<float>(d);
  float q = 0.0f;
#pragma unroll
  for (int i = 0; i < MAXV; ++i) {
    const int k = lane + i * 32;
    if (k < nv) {
      const float a = v[i].x - mean, b = v[i].y - mean, c = v[i].z - mean, e = v[i].w - mean;
      q += (a * a + b * b) + (c * c + e * e);
    }
  }
  const float rstd = rsqrtf(warp_sum(q) / static_cast<float>(d) + eps);
  const bool own_task = (row / T) == (row0 / T);
  const float4* shift = ln_smem;
  const float4* scale = ln_smem + nv;
  if (!own_task) {
    const float* base = mod_base(row);
    shift = reinterpret_cast<const float4*>(base + shift_off);
    scale = reinterpret_cast<const float4*>(base + scale_off);
  }
  uint2* yr = reinterpret_cast<uint2*>(y + static_cast<int64_t>(row) * d);
#pragma unroll
  for (int i = 0; i < MAXV; ++i) {
    const int k = lane + i * 32;
    if (k < nv) {
      const float4 sh = shift[k], sc = scale[k];
      uint2 o;
      o.x = pack_bf16x2((v[i].x - mean) * rstd * (1.0f + sc.x) + sh.x,
                        (v[i].y - mean) * rstd * (1.0f + sc.y) + sh.y);
      o.y = pack_bf16x2((v[i].z - mean) * rstd * (1.0f + sc.z) + sh.z,
                        (v[i].w - mean) * rstd * (1.0f + sc.w) + sh.w);
      yr[k] = o;
    }
  }
}

// The same LayerNorm for wide rows (d > 2048): ROWW warps share a row, each
// holding up to MAXV float4 per lane (interleaved, so every warp load is 512
// contiguous bytes), and the row's partial sums meet in shared memory in a
// fixed order (deterministic).  One warp per row would need 40 float4 per lane
// at d = 5120, which leaves one CTA per SM.
template <int MAXV, int ROWW>
__global__ void __launch_bounds__(LN_WARPS * 32)
    ln_mod_wide_kernel(const float* __restrict__ h, __nv_bfloat16* __restrict__ y, int M, int d,
                       int T, const TaskDev* __restrict__ tasks, const float* __restrict__ table,
                       int use_fmod, int block, int shift_off, int scale_off, float eps) {
  extern __shared__ float4 ln_smem[];  // [2][d / 4]: shift, scale
  __shared__ float red[2][LN_WARPS];
  constexpr int RPC = LN_WARPS / ROWW;  // rows per CTA
  pdl_trigger();
  pdl_wait();  // h is the previous kernel's output
  const int warp = warp_id(), lane = lane_id();
  const int row0 = blockIdx.x * RPC;
  const int row = row0 + warp / ROWW;
  const int part = warp % ROWW;
  const int nv = d >> 2;
  auto mod_base = [&](int r) {
    const TaskDev& t = tasks[r / T];
    return table + (use_fmod ? static_cast<int64_t>(t.fmod0)
                             : static_cast<int64_t>(t.mod0) + static_cast<int64_t>(block) * 6 * d);
  };
  float4 v[MAXV];
  float s = 0.0f;
  if (row < M) {
    const float4* hr = reinterpret_cast<const float4*>(h + static_cast<int64_t>(row) * d);
#pragma unroll
    for (int i = 0; i < MAXV; ++i) {
      const int k = part * 32 + lane + i * 32 * ROWW;
      if (k < nv) {
        v[i] = __ldcs(hr + k);
        s += (v[i].x + v[i].y) + (v[i].z + v[i].w);
      }
    }
  }
  {
    const float* base = mod_base(row0);
    const float4* shift = reinterpret_cast<const float4*>(base + shift_off);
    const float4* scale = reinterpret_cast<const float4*>(base + scale_off);
    for (int k = threadIdx.x; k < nv; k += LN_WARPS * 32) {
      ln_smem[k] = __ldg(shift + k);
      ln_smem[nv + k] = __ldg(scale + k);
    }
  }
  s = warp_sum(s);
  if (lane == 0) red[0][warp] = s;
  __syncthreads();
  float tot = 0.0f;
#pragma unroll
  for (int w = 0; w < ROWW; ++w) tot += red[0][(warp / ROWW) * ROWW + w];
  const float mean = tot / static_cast<float>(d);
  float q = 0.0f;
#pragma unroll
  for (int i = 0; i < MAXV; ++i) {
    const int k = part * 32 + lane + i * 32 * ROWW;
    if (row < M && k < nv) {
      const float a = v[i].x - mean, b = v[i].y - mean, c = v[i].z - mean, e = v[i].w - mean;
      q += (a * a + b * b) + (c * c + e * e);
    }
  }
  q = warp_sum(q);
  if (lane == 0) red[1][warp] = q;
  __syncthreads();
  if (row >= M) return;
  float qt = 0.0f;
#pragma unroll
  for (int w = 0; w < ROWW; ++w) qt += red[1][(warp / ROWW) * ROWW + w];
  const float rstd = rsqrtf(qt / static_cast<float>(d) + eps);
  const bool own_task = (row / T) == (row0 / T);
  const float4* shift = ln_smem;
  const float4* scale = ln_smem + nv;
  if (!own_task) {
    const float* base = mod_base(row);
    shift = reinterpret_cast<const float4*>(base + shift_off);
    scale = reinterpret_cast<const float4*>(base + scale_off);
  }
  uint2* yr = reinterpret_cast<uint2*>(y + static_cast<int64_t>(row) * d);
#pragma unroll
  for (int i = 0; i < MAXV; ++i) {
    const int k = part * 32 + lane + i * 32 * ROWW;
    if (k < nv) {
      const float4 sh = shift[k], sc = scale[k];
      uint2 o;
      o.x = pack_bf16x2((v[i].x - mean) * rstd * (1.0f + sc.x) + sh.x,
                        (v[i].y - mean) * rstd * (1.0f + sc.y) + sh.y);
      o.y = pack_bf16x2((v[i].z - mean) * rstd * (1.0f + sc.z) + sh.z,
                        (v[i].w - mean) * rstd * (1.0f + sc.w) + sh.w);
      yr[k] = o;
    }
  }
}

// h[r][n] = sum_k x[r][k] W_in[n][k] + b_in[n] in f32 (K = C is small).  CTA
// tile: 32 rows x 256 columns, K in chunks of 32 staged in shared memory;
// each thread accumulates 8 rows x 4 columns, so a k-step costs 8 broadcast
// reads of x and one 16-byte read of W for 32 FMAs (the kernel is bound by
// the FMA pipe and the write of h), and writes float4 rows.
constexpr int IP_ROWS = 32, IP_COLS = 256, IP_KC = 32, IP_THREADS = 256;
constexpr int IP_RG = 8, IP_CG = 4;  // rows, columns per thread
__global__ void __launch_bounds__(IP_THREADS)
    in_proj_kernel(const float* __restrict__ state, const __nv_bfloat16* __restrict__ w_in,
                   const float* __restrict__ b_in, float* __restrict__ h, int M, int d, int C,
                   int T, const TaskDev* __restrict__ tasks) {
  __shared__ float xs[IP_ROWS][IP_KC + 1];
  __shared__ __align__(16) float ws[IP_KC][IP_COLS + 4];  // padded: fewer bank conflicts on the fill
  pdl_trigger();
  pdl_wait();  // the latent state is the previous wave's output
  const int r0 = blockIdx.x * IP_ROWS;
  const int c0 = blockIdx.y * IP_COLS;
  const int tx = threadIdx.x & 63, ty = threadIdx.x >> 6;  // 64 column groups x 4 row groups
  float acc[IP_RG][IP_CG];
#pragma unroll
  for (int i = 0; i < IP_RG; ++i)
#pragma unroll
    for (int j = 0; j < IP_CG; ++j) acc[i][j] = 0.0f;
  // 16-byte loads of x (4 floats) and W (8 bf16) when C allows them
  const bool vec = (C % 8) == 0;
  for (int k0 = 0; k0 < C; k0 += IP_KC) {
    if (vec) {
      for (int idx = threadIdx.x; idx < IP_ROWS * (IP_KC / 4); idx += IP_THREADS) {
        const int rr = idx / (IP_KC / 4), kq = idx % (IP_KC / 4);
        const int row = r0 + rr, k = k0 + kq * 4;
        float4 xv = make_float4(0.f, 0.f, 0.f, 0.f);
        if (row < M && k < C) {
          const TaskDev& t = tasks[row / T];
          xv = *reinterpret_cast<const float4*>(
              state + (static_cast<int64_t>(t.state_slot) * T + (row - t.row0)) * C + k);
        }
        xs[rr][kq * 4] = xv.x;
        xs[rr][kq * 4 + 1] = xv.y;
        xs[rr][kq * 4 + 2] = xv.z;
        xs[rr][kq * 4 + 3] = xv.w;
      }
      for (int idx = threadIdx.x; idx < IP_COLS * (IP_KC / 8); idx += IP_THREADS) {
        const int nn = idx / (IP_KC / 8), kq = idx % (IP_KC / 8);
        const int col = c0 + nn, k = k0 + kq * 8;
        uint4 raw = make_uint4(0u, 0u, 0u, 0u);
        if (col < d && k < C) raw = *reinterpret_cast<const uint4*>(w_in + static_cast<int64_t>(col) * C + k);
        const __nv_bfloat162* w2 = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 f = __bfloat1622float2(w2[e]);
          ws[kq * 8 + 2 * e][nn] = f.x;
          ws[kq * 8 + 2 * e + 1][nn] = f.y;
        }
      }
    } else {
      for (int idx = threadIdx.x; idx < IP_ROWS * IP_KC; idx += IP_THREADS) {
        const int rr = idx / IP_KC, kk = idx % IP_KC;
        const int row = r0 + rr, k = k0 + kk;
        float xv = 0.0f;
        if (row < M && k < C) {
          const TaskDev& t = tasks[row / T];
          xv = state[(static_cast<int64_t>(t.state_slot) * T + (row - t.row0)) * C + k];
        }
        xs[rr][kk] = xv;
      }
      for (int idx = threadIdx.x; idx < IP_KC * IP_COLS; idx += IP_THREADS) {
        const int nn = idx / IP_KC, kk = idx % IP_KC;  // k fastest: coalesced weight rows
        const int col = c0 + nn, k = k0 + kk;
        ws[kk][nn] = (col < d && k < C) ? __bfloat162float(w_in[static_cast<int64_t>(col) * C + k]) : 0.0f;
      }
    }
    __syncthreads();
#pragma unroll 4
    for (int kk = 0; kk < IP_KC; ++kk) {
      const float4 w = *reinterpret_cast<const float4*>(&ws[kk][tx * IP_CG]);
#pragma unroll
      for (int i = 0; i < IP_RG; ++i) {
        const float xv = xs[ty * IP_RG + i][kk];
        acc[i][0] = fmaf(xv, w.x, acc[i][0]);
        acc[i][1] = fmaf(xv, w.y, acc[i][1]);
        acc[i][2] = fmaf(xv, w.z, acc[i][2]);
        acc[i][3] = fmaf(xv, w.w, acc[i][3]);
      }
    }
    __syncthreads();
  }
  const int n = c0 + tx * IP_CG;
  if (n < d) {  // d % 4 == 0, so a column group is whole
    const float4 b = *reinterpret_cast<const float4*>(b_in + n);
#pragma unroll
    for (int i = 0; i < IP_RG; ++i) {
      const int row = r0 + ty * IP_RG + i;
      if (row < M)
        *reinterpret_cast<float4*>(h + static_cast<int64_t>(row) * d + n) =
            make_float4(acc[i][0] + b.x, acc[i][1] + b.y, acc[i][2] + b.z, acc[i][3] + b.w);
    }
  }
}

// out[r][n] = act(in[r]) . W[n] + b[n] (+ add[n]).  One warp per output
// column n, all R rows at once, so each weight row is read once.
constexpr int CL_THREADS = 256;
__global__ void __launch_bounds__(CL_THREADS)
    cond_linear_kernel(const float* __restrict__ in, int R, int K,
                       const __nv_bfloat16* __restrict__ W, const float* __restrict__ b,
                       const float* __restrict__ add, float* __restrict__ out, int N,
                       int silu_in) {
  extern __shared__ float xin[];  // [R][K]
  for (int i = threadIdx.x; i < R * K; i += blockDim.x) {
    const float x = in[i];
    xin[i] = silu_in ? x / (1.0f + expf(-x)) : x;
  }
  __syncthreads();
  const int warps = blockDim.x / 32;
  const int n = blockIdx.x * warps + warp_id();
  if (n >= N) return;
  const int lane = lane_id();
  float acc[8];
#pragma unroll
  for (int r = 0; r < 8; ++r) acc[r] = 0.0f;
  const __nv_bfloat16* wr = W + static_cast<int64_t>(n) * K;
  for (int k = lane * 8; k < K; k += 256) {
    const uint4 raw = *reinterpret_cast<const uint4*>(wr + k);
    const __nv_bfloat162* w2 = reinterpret_cast<const __nv_bfloat162*>(&raw);
    float w[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __bfloat1622float2(w2[i]);
      w[2 * i] = f.x;
      w[2 * i + 1] = f.y;
    }
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      if (r < R) {
        const float* xr = xin + r * K + k;
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[r] = fmaf(xr[i], w[i], acc[r]);
      }
    }
  }
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    float v = acc[r];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == 0 && r < R) out[static_cast<int64_t>(r) * N + n] = v + b[n] + (add ? add[n] : 0.0f);
  }
}

__global__ void f32_to_bf16_kernel(const float* __restrict__ src, __nv_bfloat16* __restrict__ dst,
                                   int64_t n) {
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    dst[i] = __float2bfloat16_rn(src[i]);
}

}  // namespace

cudaError_t launch_ln_mod(const float* h, __nv_bfloat16* y, int M, int d, int T,
                          const TaskDev* tasks, const float* table, int use_fmod, int block,
                          int shift_off, int scale_off, float eps, cudaStream_t st) {
  if (M <= 0) return cudaSuccess;
  if (d % 4 != 0) return cudaErrorInvalidValue;
  const int nv = d / 4;
  const size_t smem = 2 * static_cast<size_t>(nv) * sizeof(float4);
  if (smem > 48 * 1024) return cudaErrorInvalidValue;
  const int grid = (M + LN_WARPS - 1) / LN_WARPS;
#define PSV_LN_LAUNCH(V)                                                                     \
  return launch_pdl(ln_mod_kernel<V>, dim3(grid), dim3(LN_WARPS * 32), smem, st, h, y, M, d, T, \
                    tasks, table, use_fmod, block, shift_off, scale_off, eps)
#define PSV_LN_WIDE(V, R)                                                                    \
  return launch_pdl(ln_mod_wide_kernel<V, R>, dim3((M + LN_WARPS / R - 1) / (LN_WARPS / R)),  \
                    dim3(LN_WARPS * 32), smem, st, h, y, M, d, T, tasks, table, use_fmod, block, \
                    shift_off, scale_off, eps)
  if (nv <= 32 * 1) PSV_LN_LAUNCH(1);
  else if (nv <= 32 * 2) PSV_LN_LAUNCH(2);
  else if (nv <= 32 * 4) PSV_LN_LAUNCH(4);
  else if (nv <= 32 * 8) PSV_LN_LAUNCH(8);
  else if (nv <= 32 * 12) PSV_LN_LAUNCH(12);
  else if (nv <= 32 * 16) PSV_LN_LAUNCH(16);
  else if (nv <= 2 * 32 * 12) PSV_LN_WIDE(12, 2);   // d <= 3072
  else if (nv <= 4 * 32 * 10) PSV_LN_WIDE(10, 4);   // d <= 5120
  else if (nv <= 4 * 32 * 12) PSV_LN_WIDE(12, 4);
  else if (nv <= 8 * 32 * 12) PSV_LN_WIDE(12, 8);
  else return cudaErrorInvalidValue;
#undef PSV_LN_LAUNCH
#undef PSV_LN_WIDE
  return cudaGetLastError();
}

cudaError_t launch_in_proj(const float* state, const __nv_bfloat16* w_in, const float* b_in,
                           float* h, int M, int d, int C, int T, const TaskDev* tasks,
                           cudaStream_t st) {
  if (M <= 0) return cudaSuccess;
  if (d % 4 != 0) return cudaErrorInvalidValue;
  dim3 grid((M + IP_ROWS - 1) / IP_ROWS, (d + IP_COLS - 1) / IP_COLS);
  return launch_pdl(in_proj_kernel, grid, dim3(IP_THREADS), 0, st, state, w_in, b_in, h, M, d, C, T, tasks);
}

cudaError_t launch_cond_linear(const float* in, int R, int K, const __nv_bfloat16* W,
                               const float* b, const float* add, float* out, int N, int silu_in,
                               cudaStream_t st) {
  if (R < 1 || R > 8 || K % 8 != 0) return cudaErrorInvalidValue;
  const size_t smem = static_cast<size_t>(R) * K * sizeof(float);
  static uint64_t set_up = 0;
  cudaError_t e = once_per_device(&set_up, [](int) {
    return cudaFuncSetAttribute(cond_linear_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                200 * 1024);
  });
  if (e != cudaSuccess) return e;
  if (smem > 200 * 1024) return cudaErrorInvalidValue;
  const int warps = CL_THREADS / 32;
  cond_linear_kernel<<<(N + warps - 1) / warps, CL_THREADS, smem, st>>>(in, R, K, W, b, add, out,
                                                                          N, silu_in);
  return cudaGetLastError();
}

cudaError_t launch_f32_to_bf16(const float* src, __nv_bfloat16* dst, int64_t n, cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  f32_to_bf16_kernel<<<1184, 256, 0, st>>>(src, dst, n);
  return cudaGetLastError();
}

}  // namespace psv
