// Host-side utilities shared by every entry point: the device check, CUDA error recording,
// TMA tensor-map encoding, the bounded-wait limit and the diagnostics entry points.
#include <cudaTypedefs.h>

#include <atomic>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "common.cuh"

namespace ta {

static thread_local char g_last_err[256] = "";
static std::atomic<int64_t> g_wait_limit_ns{2000000000LL};
static std::atomic<int> g_bwd_split{0};         // 0: chosen per launch from the grid size
static std::atomic<int> g_fwd_split{0};

int record_cuda(cudaError_t e) {
  if (e == cudaSuccess) return TREE_OK;
  std::snprintf(g_last_err, sizeof(g_last_err), "%s: %s", cudaGetErrorName(e), cudaGetErrorString(e));
  return TREE_ERR_CUDA;
}

int check_device() {
  static int cached[64];          // 0 unknown, 1 ok, 2 wrong arch
  int dev = 0;
  int rc = record_cuda(cudaGetDevice(&dev));
  if (rc) return rc;
  if (dev >= 0 && dev < 64 && cached[dev]) return cached[dev] == 1 ? TREE_OK : TREE_ERR_ARCH;
  int major = 0, minor = 0;
  rc = record_cuda(cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev));
  if (rc) return rc;
  rc = record_cuda(cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev));
  if (rc) return rc;
  const bool ok = (major == 10 && minor == 3);
  if (dev >= 0 && dev < 64) cached[dev] = ok ? 1 : 2;
  return ok ? TREE_OK : TREE_ERR_ARCH;
}

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 3-D map over a bf16 tensor [rows][heads][d] (d innermost), box = 64 x 1 x 128 with the
// 128-byte swizzle; out-of-range rows read as zero.
int make_tmap_bf16_3d(CUtensorMap* m, const void* base, int d, int heads, int rows) {
  auto fn = encode_fn();
  if (!fn) {
    std::snprintf(g_last_err, sizeof(g_last_err), "cuTensorMapEncodeTiled entry point unavailable");
    return TREE_ERR_CUDA;
  }
  if ((reinterpret_cast<uintptr_t>(base) & 15) != 0) return TREE_ERR_ARG;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(heads),
                        static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(heads) * d * 2};
  cuuint32_t box[3] = {64, 1, TILE};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    std::snprintf(g_last_err, sizeof(g_last_err), "cuTensorMapEncodeTiled failed (CUresult %d)", (int)r);
    return TREE_ERR_CUDA;
  }
  return TREE_OK;
}

// 2-D map over an fp32 matrix [rows][inner] (inner contiguous), unswizzled box
// box_inner x box_rows (used as the target of TMA reduce-add).
int make_tmap_f32_2d(CUtensorMap* m, const void* base, int inner, int rows, int box_inner, int box_rows) {
  auto fn = encode_fn();
  if (!fn) {
    std::snprintf(g_last_err, sizeof(g_last_err), "cuTensorMapEncodeTiled entry point unavailable");
    return TREE_ERR_CUDA;
  }
  if ((reinterpret_cast<uintptr_t>(base) & 15) != 0 || (inner * 4) % 16 != 0) return TREE_ERR_ARG;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(inner) * 4};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(box_inner), static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    std::snprintf(g_last_err, sizeof(g_last_err), "cuTensorMapEncodeTiled (f32) failed (CUresult %d)", (int)r);
    return TREE_ERR_CUDA;
  }
  return TREE_OK;
}

// 2-D map over a bf16 matrix [rows][inner] (inner contiguous), unswizzled box box_inner x
// box_rows; rows outside [0, rows) and columns past inner read as zero.
int make_tmap_bf16_2d(CUtensorMap* m, const void* base, int inner, int rows, int box_inner, int box_rows) {
  auto fn = encode_fn();
  if (!fn) {
    std::snprintf(g_last_err, sizeof(g_last_err), "cuTensorMapEncodeTiled entry point unavailable");
    return TREE_ERR_CUDA;
  }
  if ((reinterpret_cast<uintptr_t>(base) & 15) != 0 || (inner * 2) % 16 != 0) return TREE_ERR_ARG;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(inner) * 2};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(box_inner), static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    std::snprintf(g_last_err, sizeof(g_last_err), "cuTensorMapEncodeTiled (bf16 2-D) failed (CUresult %d)", (int)r);
    return TREE_ERR_CUDA;
  }
  return TREE_OK;
}

// 2-D map over a bf16 matrix [rows][inner] with the 128-byte swizzle (box_inner x 2 B <= 128),
// the layout tcgen05 shared-memory descriptors read; out-of-range elements read as zero.
int make_tmap_bf16_2d_sw128(CUtensorMap* m, const void* base, int inner, int rows, int box_inner, int box_rows) {
  auto fn = encode_fn();
  if (!fn) {
    std::snprintf(g_last_err, sizeof(g_last_err), "cuTensorMapEncodeTiled entry point unavailable");
    return TREE_ERR_CUDA;
  }
  if ((reinterpret_cast<uintptr_t>(base) & 15) != 0 || (inner * 2) % 16 != 0) return TREE_ERR_ARG;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(inner) * 2};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(box_inner), static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    std::snprintf(g_last_err, sizeof(g_last_err), "cuTensorMapEncodeTiled (bf16 2-D sw128) failed (CUresult %d)",
                  (int)r);
    return TREE_ERR_CUDA;
  }
  return TREE_OK;
}

static cudaEvent_t g_events[4];
static int g_n_events = 0;

void record_timing_event(int i, cudaStream_t s) {
  if (i < g_n_events && g_events[i]) cudaEventRecord(g_events[i], s);
}

uint64_t wait_limit_ns() { return static_cast<uint64_t>(g_wait_limit_ns.load()); }
int bwd_split_override() { return g_bwd_split.load(); }
int fwd_split_override() { return g_fwd_split.load(); }

int plan_ok(const tree_plan_t* p) {
  if (!p || !p->tok_in || !p->row_ptr || !p->row_idx || !p->col_ptr || !p->col_idx || !p->tile_class ||
      !p->row_order || !p->col_order || !p->pos)
    return TREE_ERR_ARG;
  if (p->n_tokens <= 0 || p->n_tiles != (p->n_tokens + TILE - 1) / TILE || p->n_paths <= 0)
    return TREE_ERR_SHAPE;
  return TREE_OK;
}

// ------------------------------------------------------------------------------------------
// self-test of the bounded wait: one warp waits on a barrier that nothing arrives at
__global__ void k_selftest_timeout(int32_t* status, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&bar, 1);
  }
  __syncthreads();
  WaitCtl wc{&abort_flag, status, limit_ns};
  if (threadIdx.x == 0) mbar_wait(&bar, 0, wc);
  __syncthreads();
}

}  // namespace ta

using namespace ta;

extern "C" {

int tree_set_timing_events(void* const* events, int n) {
  if (n < 0 || n > 4 || (n > 0 && !events)) return TREE_ERR_ARG;
  for (int i = 0; i < 4; ++i) g_events[i] = i < n ? static_cast<cudaEvent_t>(events[i]) : nullptr;
  g_n_events = n;
  return TREE_OK;
}

int tree_set_fwd_split(int split) {
  if (split != 0 && split != 1 && split != 2 && split != 4) return TREE_ERR_ARG;
  g_fwd_split.store(split);
  return TREE_OK;
}

int tree_set_bwd_split(int split) {
  if (split != 0 && split != 1 && split != 2 && split != 4) return TREE_ERR_ARG;
  g_bwd_split.store(split);
  return TREE_OK;
}

int tree_set_wait_limit_ns(int64_t ns) {
  if (ns < 100000) ns = 100000;
  g_wait_limit_ns.store(ns);
  return TREE_OK;
}

int tree_selftest_timeout(int32_t* status_dev, int64_t ns, tree_stream_t stream) {
  if (!status_dev) return TREE_ERR_ARG;
  int rc = check_device();
  if (rc) return rc;
  if (ns < 1000) ns = 1000;
  k_selftest_timeout<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(status_dev, (uint64_t)ns);
  return record_cuda(cudaGetLastError());
}

const char* tree_strerror(int code) {
  switch (code) {
    case TREE_OK: return "ok";
    case TREE_ERR_INVALID_TREE: return "invalid tree (parent out of range, cycle, no root, negative length or bad token total)";
    case TREE_ERR_SHAPE: return "unsupported shape (d must be 64 or 128, Hq % Hkv == 0, plan/tensor mismatch)";
    case TREE_ERR_ARCH: return "the current device is not compute capability 10.3 (GB300)";
    case TREE_ERR_CUDA: return "CUDA runtime error (see tree_last_cuda_error)";
    case TREE_ERR_TIMEOUT: return "a bounded device wait expired";
    case TREE_ERR_ARG: return "null or misaligned pointer, or bad size";
    case TREE_ERR_SCRATCH: return "problem needs more scratch than the non-allocating backward's fixed array";
    default: return "unknown error code";
  }
}

const char* tree_last_cuda_error(void) { return g_last_err; }

int tree_version(void) { return 1; }

}  // extern "C"
