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

// The LayerNorm of rows of up to 2048 values, staged by bulk copies: one
// persistent CTA per SM takes a contiguous block of rows (so the rows of at
// most two tasks: their shift / scale vectors are copied to shared memory
// first), brought in by cp.async.bulk in batches of half the staging area,
// the next batch's copies in flight while 16 warps normalise the current one
// (one row per warp, in registers).  Every row is computed with the order of
// operations of ln_mod_kernel, so the two kernels give the same bits.
constexpr int LNB_WARPS = 16;
constexpr uint32_t LNB_SMEM = 200 * 1024;

__device__ __forceinline__ void bulk_load_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

template <int MAXV>
__global__ void __launch_bounds__(LNB_WARPS * 32, 1)
    ln_bulk_kernel(const float* __restrict__ h, __nv_bfloat16* __restrict__ y, int M, int d, int T,
                   const TaskDev* __restrict__ tasks, const float* __restrict__ table, int use_fmod,
                   int block, int shift_off, int scale_off, float eps, int* err) {
  extern __shared__ __align__(128) uint8_t lnb_smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(lnb_smem);          // [2]
  float4* tab = reinterpret_cast<float4*>(lnb_smem + 128);           // [task a, b][shift, scale][d / 4]
  const int warp = warp_id(), lane = lane_id();
  const int nv = d >> 2;
  const uint32_t row_bytes = static_cast<uint32_t>(d) * 4;
  uint8_t* rows_area = lnb_smem + 128 + 4 * row_bytes;
  const uint32_t half = ((LNB_SMEM - 128 - 4 * row_bytes) / 2) & ~15u;
  if (threadIdx.x == 0) {
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    fence_mbar_init();
  }
  pdl_trigger();
  pdl_wait();  // h is the previous kernel's output
  __syncthreads();
  const int per = (M + static_cast<int>(gridDim.x) - 1) / static_cast<int>(gridDim.x);
  const int r0 = min(M, static_cast<int>(blockIdx.x) * per), r1 = min(M, r0 + per);
  if (r0 >= r1) return;
  const int batch = static_cast<int>(half / row_bytes);
  const int nbatch = (r1 - r0 + batch - 1) / batch;
  auto vec_base = [&](int ti) {
    const TaskDev& t = tasks[ti];
    return table + (use_fmod ? static_cast<int64_t>(t.fmod0)
                             : static_cast<int64_t>(t.mod0) + static_cast<int64_t>(block) * 6 * d);
  };
  auto issue = [&](int k) {
    const int b0 = r0 + k * batch, nb = min(batch, r1 - b0);
    uint8_t* buf = rows_area + (k & 1) * half;
    mbar_arrive_expect_tx(&bars[k & 1], static_cast<uint32_t>(nb) * row_bytes);
    for (int i = 0; i < nb; ++i)
      bulk_load_g2s(buf + i * row_bytes, h + static_cast<int64_t>(b0 + i) * d, row_bytes, &bars[k & 1]);
  };
  if (threadIdx.x == 0) issue(0);
  const int ta = r0 / T, tb = (r1 - 1) / T;
  for (int idx = threadIdx.x; idx < 4 * nv; idx += LNB_WARPS * 32) {
    const int which = idx / nv, c = idx - which * nv;  // which: task (bit 1), scale (bit 0)
    tab[idx] = __ldg(reinterpret_cast<const float4*>(vec_base((which & 2) ? tb : ta) +
                                                     ((which & 1) ? scale_off : shift_off)) + c);
  }
  int issued = 1;
  bool ok = true;
  for (int k = 0; k < nbatch; ++k) {
    if (k + 1 < nbatch) {
      if (threadIdx.x == 0) {  // buffer (k+1)&1 was released at the end of batch k-1
        fence_proxy_async_smem();
        issue(k + 1);
      }
      ++issued;
    }
    // (the first wait also orders the table fill above before its use)
    ok = __syncthreads_and(mbar_wait(&bars[k & 1], (k >> 1) & 1, err, ERR_LN_TIMEOUT) ? 1 : 0) != 0;
    if (!ok) break;
    const int b0 = r0 + k * batch, nb = min(batch, r1 - b0);
    const uint8_t* buf = rows_area + (k & 1) * half;
    for (int i = warp; i < nb; i += LNB_WARPS) {
      const int row = b0 + i;
      const float4* hr = reinterpret_cast<const float4*>(buf + i * row_bytes);
      float4 v[MAXV];
      float s = 0.0f;
#pragma unroll
      for (int j = 0; j < MAXV; ++j) {
        const int c = lane + j * 32;
        if (c < nv) {
          v[j] = hr[c];
          s += (v[j].x + v[j].y) + (v[j].z + v[j].w);
        }
      }
      const float mean = warp_sum(s) / static_cast<float>(d);
      float q = 0.0f;
#pragma unroll
      for (int j = 0; j < MAXV; ++j) {
        const int c = lane + j * 32;
        if (c < nv) {
          const float a = v[j].x - mean, b = v[j].y - mean, cc = v[j].z - mean, e = v[j].w - mean;
          q += (a * a + b * b) + (cc * cc + e * e);
        }
      }
      const float rstd = rsqrtf(warp_sum(q) / static_cast<float>(d) + eps);
      const int ti = row / T;
      const float4* shift = tab + (ti == ta ? 0 : 2) * nv;
      const float4* scale = shift + nv;
      if (ti != ta && ti != tb) {  // only when a CTA's rows span more than two tasks
        shift = reinterpret_cast<const float4*>(vec_base(ti) + shift_off);
        scale = reinterpret_cast<const float4*>(vec_base(ti) + scale_off);
      }
      uint2* yr = reinterpret_cast<uint2*>(y + static_cast<int64_t>(row) * d);
#pragma unroll
      for (int j = 0; j < MAXV; ++j) {
        const int c = lane + j * 32;
        if (c < nv) {
          const float4 sh = shift[c], sc = scale[c];
          uint2 o;
          o.x = pack_bf16x2((v[j].x - mean) * rstd * (1.0f + sc.x) + sh.x,
                            (v[j].y - mean) * rstd * (1.0f + sc.y) + sh.y);
          o.y = pack_bf16x2((v[j].z - mean) * rstd * (1.0f + sc.z) + sh.z,
                            (v[j].w - mean) * rstd * (1.0f + sc.w) + sh.w);
          yr[c] = o;
        }
      }
    }
    __syncthreads();  // batch k's buffer is refilled by batch k + 2
  }
  if (!ok && threadIdx.x == 0) {
    // Let this CTA's copies still in flight land before it leaves (bounded).
    const uint64_t t0 = global_timer_ns();
    for (int k = 0; k < issued; ++k)
      while (!mbar_try_wait(&bars[k & 1], (k >> 1) & 1) && global_timer_ns() - t0 < kWaitLimitNs) {
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

// Split of the latent rows for the tensor-core in-projection: row r of the
// wave (task r / T, token r % T) -> [bf16(x) | bf16(x - bf16(x)) | 0 ...].
// x - bf16(x) is exact in f32, so hi + lo carries x to within 2^-16 relative.
__global__ void in_split_kernel(const float* __restrict__ state, const TaskDev* __restrict__ tasks,
                                __nv_bfloat16* __restrict__ xs, int M, int C, int T, int K2) {
  pdl_trigger();
  pdl_wait();  // the latent state is the previous wave's output
  const int64_t total = static_cast<int64_t>(M) * K2;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int r = static_cast<int>(i / K2), k = static_cast<int>(i % K2);
    float v = 0.0f;
    if (k < 2 * C) {
      const TaskDev& t = tasks[r / T];
      const float x = state[(static_cast<int64_t>(t.state_slot) * T + (r - t.row0)) * C + (k % C)];
      const float hi = __bfloat162float(__float2bfloat16_rn(x));
      v = k < C ? hi : x - hi;
    }
    xs[i] = __float2bfloat16_rn(v);
  }
}

__global__ void build_in2_kernel(const __nv_bfloat16* __restrict__ w_in, __nv_bfloat16* __restrict__ w2,
                                 int d, int C, int K2, int rows) {
  const int64_t total = static_cast<int64_t>(rows) * K2;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int n = static_cast<int>(i / K2), k = static_cast<int>(i % K2);
    w2[i] = (n < d && k < 2 * C) ? w_in[static_cast<int64_t>(n) * C + (k % C)] : __float2bfloat16_rn(0.0f);
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
                          int shift_off, int scale_off, float eps, int* err, cudaStream_t st) {
  if (M <= 0) return cudaSuccess;
  if (d % 4 != 0) return cudaErrorInvalidValue;
  const int nv = d / 4;
  if (d <= 2048 && err) {
    static uint64_t set_up = 0;
    static int sms[64] = {};
    cudaError_t e = once_per_device(&set_up, [&](int dev) {
      cudaError_t r = cudaDeviceGetAttribute(&sms[dev], cudaDevAttrMultiProcessorCount, dev);
      if (r != cudaSuccess) return r;
#define PSV_LNB_ATTR(V)                                                                        \
  if ((r = cudaFuncSetAttribute(ln_bulk_kernel<V>, cudaFuncAttributeMaxDynamicSharedMemorySize, \
                                static_cast<int>(LNB_SMEM))) != cudaSuccess)                    \
    return r;
      PSV_LNB_ATTR(4) PSV_LNB_ATTR(8) PSV_LNB_ATTR(12) PSV_LNB_ATTR(16)
#undef PSV_LNB_ATTR
      return cudaSuccess;
    });
    if (e != cudaSuccess) return e;
    int dev = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    const int grid = M < sms[dev] ? M : sms[dev];
#define PSV_LNB_LAUNCH(V)                                                                   \
  return launch_pdl(ln_bulk_kernel<V>, dim3(grid), dim3(LNB_WARPS * 32), LNB_SMEM, st, h, y, M, d, \
                    T, tasks, table, use_fmod, block, shift_off, scale_off, eps, err)
    if (nv <= 32 * 4) PSV_LNB_LAUNCH(4);
    else if (nv <= 32 * 8) PSV_LNB_LAUNCH(8);
    else if (nv <= 32 * 12) PSV_LNB_LAUNCH(12);
    else PSV_LNB_LAUNCH(16);
#undef PSV_LNB_LAUNCH
  }
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

cudaError_t launch_in_split(const float* state, const TaskDev* tasks, __nv_bfloat16* xs, int M,
                            int C, int T, int K2, cudaStream_t st) {
  if (M <= 0) return cudaSuccess;
  const int64_t total = static_cast<int64_t>(M) * K2;
  const int grid = static_cast<int>((total + 255) / 256 < 1216 ? (total + 255) / 256 : 1216);
  return launch_pdl(in_split_kernel, dim3(grid), dim3(256), 0, st, state, tasks, xs, M, C, T, K2);
}

cudaError_t launch_build_in2(const __nv_bfloat16* w_in, __nv_bfloat16* w_in2, int d, int C,
                             int K2, int rows, cudaStream_t st) {
  const int64_t total = static_cast<int64_t>(rows) * K2;
  const int grid = static_cast<int>((total + 255) / 256 < 1216 ? (total + 255) / 256 : 1216);
  build_in2_kernel<<<grid, 256, 0, st>>>(w_in, w_in2, d, C, K2, rows);
  return cudaGetLastError();
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
