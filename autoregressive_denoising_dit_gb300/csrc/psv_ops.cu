// Kernel-level entry points of libpsv: the wave's window attention as a
// standalone call on caller buffers (include/psv.h, "kernel-level window
// attention").  It launches the same attention kernel the wave uses.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstring>
#include <mutex>

#include "../../include/psv.h"
#include "psv_device.cuh"
#include "psv_kernels.h"

#define PSV_API extern "C" __attribute__((visibility("default")))

using psv::TaskDev;

namespace {

size_t up256(size_t x) { return (x + 255) / 256 * 256; }

// Scratch layout: [error word | task table | arrival counters | partials].
struct AttnScratch {
  size_t err, tasks, counters, part, total;
};

AttnScratch attn_scratch_layout(const psv_attn_problem& p) {
  AttnScratch s{};
  s.err = 0;
  s.tasks = 256;
  s.counters = s.tasks + up256(sizeof(TaskDev) * static_cast<size_t>(p.n));
  s.part = s.counters + up256(sizeof(int) * psv::attn_counter_ints(p.n, p.T, p.H));
  s.total = s.part + up256(psv::attn_part_floats(p.n, p.T, p.H, p.dh) * sizeof(float));
  return s;
}

bool attn_problem_ok(const psv_attn_problem* p) {
  if (!p) return false;
  if (p->n < 1 || p->T < 1 || p->H < 1 || p->L < 1) return false;
  if (p->dh != 32 && p->dh != 64 && p->dh != 128) return false;
  if ((p->H * p->dh) % 8 != 0) return false;
  if (p->k_rows < p->L || p->vt_cols < p->L || p->vt_cols % 8 != 0) return false;
  const int64_t rows = static_cast<int64_t>(p->n) * p->T;
  if (rows > (1 << 28) || static_cast<int64_t>(p->n) * p->k_rows > (1ll << 31)) return false;
  return true;
}

bool aligned16(const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15) == 0; }

}  // namespace

// Enqueue one attention call with the given scratch (shared by the call with
// caller scratch and any other front end of the same kernel).
int psv_attention_enqueue(const psv_attn_problem* p, const void* q, const void* k, const void* vt,
                          void* o, char* scratch, cudaStream_t st) {
  const AttnScratch L = attn_scratch_layout(*p);
  const int d = p->H * p->dh;
  const uint32_t aw = p->dh < 64 ? p->dh : 64;
  const CUtensorMapSwizzle swq = aw == 32 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B;
  CUtensorMap tmQ, tmK, tmV;
  bool ok = true;
  {
    uint64_t dims[2] = {static_cast<uint64_t>(d), static_cast<uint64_t>(p->n) * p->T};
    uint64_t str[1] = {static_cast<uint64_t>(d) * 2};
    uint32_t box[2] = {aw, 128};
    ok &= psv::encode_bf16_map(&tmQ, 2, const_cast<void*>(q), dims, str, box, swq);
  }
  {
    uint64_t dims[3] = {static_cast<uint64_t>(d), static_cast<uint64_t>(p->k_rows),
                        static_cast<uint64_t>(p->n)};
    uint64_t str[2] = {static_cast<uint64_t>(d) * 2, static_cast<uint64_t>(d) * 2 * p->k_rows};
    uint32_t box[3] = {aw, psv::attn_k_box_rows(), 1};
    ok &= psv::encode_bf16_map(&tmK, 3, const_cast<void*>(k), dims, str, box, swq);
  }
  {
    uint64_t dims[3] = {static_cast<uint64_t>(p->vt_cols), static_cast<uint64_t>(p->dh),
                        static_cast<uint64_t>(p->n) * p->H};
    uint64_t str[2] = {static_cast<uint64_t>(p->vt_cols) * 2,
                       static_cast<uint64_t>(p->vt_cols) * 2 * p->dh};
    uint32_t box[3] = {64, psv::attn_v_box_rows(p->dh), 1};
    ok &= psv::encode_bf16_map(&tmV, 3, const_cast<void*>(vt), dims, str, box,
                               CU_TENSOR_MAP_SWIZZLE_128B);
  }
  if (!ok) return PSV_EINVAL;
  cudaError_t e;
  // The error word and the counters must start at zero.
  if ((e = cudaMemsetAsync(scratch + L.err, 0, sizeof(int), st)) != cudaSuccess) return PSV_ECUDA;
  if ((e = cudaMemsetAsync(scratch + L.counters, 0, sizeof(int) * psv::attn_counter_ints(p->n, p->T, p->H),
                           st)) != cudaSuccess)
    return PSV_ECUDA;
  TaskDev* tasks = reinterpret_cast<TaskDev*>(scratch + L.tasks);
  if ((e = psv::launch_fill_attn_tasks(tasks, p->n, p->T, p->L, st)) != cudaSuccess) return PSV_ECUDA;
  psv::AttnParams a{};
  a.T = p->T;
  a.d = d;
  a.dh = p->dh;
  a.H = p->H;
  a.S = 1;
  a.Lr = p->k_rows;
  a.Lp = p->vt_cols;
  a.block = 0;
  a.n_tasks = p->n;
  a.tasks = tasks;
  a.o = static_cast<__nv_bfloat16*>(o);
  a.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(p->dh)));
  a.part = reinterpret_cast<float*>(scratch + L.part);
  a.counters = reinterpret_cast<int*>(scratch + L.counters);
  a.max_pairs = psv::attn_units(p->T);
  a.err = reinterpret_cast<int*>(scratch + L.err);
  a.n_pieces = psv::attn_pieces_uniform(p->L, p->n, p->T, p->H);
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return PSV_ECUDA;
  const int grid = psv::attn_grid_size(a.n_pieces, sms);
  if ((e = psv::launch_attention(&tmQ, &tmK, &tmV, a, p->n, grid, st)) != cudaSuccess) return PSV_ECUDA;
  return PSV_OK;
}

PSV_API int psv_attention_scratch_bytes(const psv_attn_problem* p, size_t* bytes) {
  if (!attn_problem_ok(p) || !bytes) return PSV_EINVAL;
  *bytes = attn_scratch_layout(*p).total;
  return PSV_OK;
}

PSV_API int psv_attention(const psv_attn_problem* p, const void* q, const void* k, const void* vt,
                          void* o, void* scratch, size_t scratch_bytes, void* cuda_stream) {
  if (!attn_problem_ok(p)) return PSV_EINVAL;
  if (!q || !k || !vt || !o || !scratch) return PSV_EINVAL;
  if (!aligned16(q) || !aligned16(k) || !aligned16(vt) || !aligned16(o)) return PSV_EINVAL;
  if ((reinterpret_cast<uintptr_t>(scratch) & 255) != 0) return PSV_EINVAL;
  if (scratch_bytes < attn_scratch_layout(*p).total) return PSV_EINVAL;
  return psv_attention_enqueue(p, q, k, vt, o, static_cast<char*>(scratch),
                               static_cast<cudaStream_t>(cuda_stream));
}

// ---------------------------------------------------------------------------
// Allocation-free variant.  Some callers cannot allocate device memory when
// they call: a control loop that must never enter the CUDA allocator after
// start-up (its latency and failure modes are not bounded), or a host
// framework that owns every device allocation and hands out no scratch.  For
// them the scratch of the attention call lives in this file-scope array.
// The CUDA module that holds it is loaded on a device, and the array
// reserved there until the process exits, when the module is first used on
// that device: with CUDA's default lazy module loading that is the set-up of
// the first call below.  Nothing on the call path allocates host or device
// memory after that set-up.
namespace {

constexpr size_t kNoAllocScratchBytes = PSV_ATTN_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_attn_scratch[kNoAllocScratchBytes];

std::mutex g_scratch_mu;
char* g_scratch_ptr[64] = {};  // device address of g_attn_scratch, per device

// Device address of the array on the current device, looked up once per
// device with that device current: in host code the name g_attn_scratch is
// only a host-side stand-in, which a kernel must never be given.
int noalloc_scratch(char** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return PSV_ECUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_attn_scratch) != cudaSuccess || !ptr) return PSV_ECUDA;
    g_scratch_ptr[dev] = static_cast<char*>(ptr);
  }
  *out = g_scratch_ptr[dev];
  return PSV_OK;
}

}  // namespace

PSV_API int psv_attention_noalloc(const psv_attn_problem* p, const void* q, const void* k,
                                  const void* vt, void* o, void* cuda_stream) {
  if (!attn_problem_ok(p)) return PSV_EINVAL;
  if (!q || !k || !vt || !o) return PSV_EINVAL;
  if (!aligned16(q) || !aligned16(k) || !aligned16(vt) || !aligned16(o)) return PSV_EINVAL;
  if (attn_scratch_layout(*p).total > kNoAllocScratchBytes) return PSV_ENOMEM;  // over the fixed size
  char* scratch = nullptr;
  if (int r = noalloc_scratch(&scratch)) return r;
  return psv_attention_enqueue(p, q, k, vt, o, scratch, static_cast<cudaStream_t>(cuda_stream));
}

PSV_API int psv_attention_noalloc_status(int* status, void* cuda_stream) {
  if (!status) return PSV_EINVAL;
  char* scratch = nullptr;
  if (int r = noalloc_scratch(&scratch)) return r;
  const cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  // The error word sits at the start of the array (offset 0 of the layout).
  if (cudaStreamSynchronize(st) != cudaSuccess) return PSV_ECUDA;
  if (cudaMemcpy(status, scratch, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return PSV_ECUDA;
  return PSV_OK;
}
