// RoPE at tree-depth positions ("Tree Training 技术详解", section 5) and the per-token loss
// weight g_t/K applied to an upstream gradient (section 6.2).  Both are HBM-bound streaming
// kernels: 16-byte vector loads/stores, angles computed once per token and shared by heads.
#include "common.cuh"

namespace ta {
namespace {

constexpr int kRopeTok = 8;          // tokens per block
constexpr int kRopeThreads = 256;

// One block rotates every head of kRopeTok consecutive tokens.  Work item = (token, head,
// 8-wide vector v of the first half); it reads x[c..c+7] and x[c+d/2..c+d/2+7], c = 8v.
template <int HD>
__global__ void __launch_bounds__(kRopeThreads) k_rope(const int32_t* __restrict__ pos, int N, float theta,
                                                       const uint4* q, uint4* qr, int Hq, const uint4* k,
                                                       uint4* kr, int Hkv) {
  constexpr int HALF = HD / 2;
  constexpr int VPR = HALF / 8;                       // vectors per half row
  __shared__ float s_cos[kRopeTok][HALF], s_sin[kRopeTok][HALF];
  const int t0 = blockIdx.x * kRopeTok;
  for (int e = threadIdx.x; e < kRopeTok * HALF; e += blockDim.x) {
    const int tt = e / HALF, c = e % HALF;
    const int t = t0 + tt;
    const float ang = (t < N ? static_cast<float>(pos[t]) : 0.f) * rope_inv_freq(c, HD, theta);
    float sv, cv;
    sincosf(ang, &sv, &cv);
    s_cos[tt][c] = cv;
    s_sin[tt][c] = sv;
  }
  __syncthreads();
  const int H = Hq + Hkv;
  const int items = kRopeTok * H * VPR;
  for (int it = threadIdx.x; it < items; it += blockDim.x) {
    const int v = it % VPR;
    const int hh = (it / VPR) % H;
    const int tt = it / (VPR * H);
    const int t = t0 + tt;
    if (t >= N) continue;
    const uint4* src;
    uint4* dst;
    size_t row;
    if (hh < Hq) { row = (size_t)t * Hq + hh; src = q; dst = qr; }
    else { row = (size_t)t * Hkv + (hh - Hq); src = k; dst = kr; }
    const size_t base = row * (HD / 8);                // in 16-byte vectors
    const uint4 a = src[base + v], b = src[base + VPR + v];
    const uint32_t av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
    uint32_t oa[4], ob[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int c = v * 8 + 2 * e;
      const float x1l = bf16lo(av[e]), x1h = bf16hi(av[e]);
      const float x2l = bf16lo(bv[e]), x2h = bf16hi(bv[e]);
      const float cl = s_cos[tt][c], ch = s_cos[tt][c + 1], sl = s_sin[tt][c], sh = s_sin[tt][c + 1];
      oa[e] = pack_bf16(x1l * cl - x2l * sl, x1h * ch - x2h * sh);
      ob[e] = pack_bf16(x2l * cl + x1l * sl, x2h * ch + x1h * sh);
    }
    dst[base + v] = make_uint4(oa[0], oa[1], oa[2], oa[3]);
    dst[base + VPR + v] = make_uint4(ob[0], ob[1], ob[2], ob[3]);
  }
}

// dO[t][h][:] = w[t] * U[t][h][:], 8 bf16 per thread
__global__ void k_apply_weights(const float* __restrict__ w, const uint4* u, uint4* out, int N, int row_vecs,
                                 int per_token) {
  const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  const size_t total = (size_t)N * per_token;
  if (i >= total) return;
  const int t = static_cast<int>(i / per_token);
  const float wt = w[t];
  const uint4 a = u[i];
  const uint32_t av[4] = {a.x, a.y, a.z, a.w};
  uint32_t o[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) o[e] = pack_bf16(wt * bf16lo(av[e]), wt * bf16hi(av[e]));
  out[i] = make_uint4(o[0], o[1], o[2], o[3]);
  (void)row_vecs;
}

// dst[r] = src[rows[r]] for bf16 rows of row_elems elements (a multiple of 8), 16 bytes a thread
__global__ void k_gather_rows(const int32_t* __restrict__ rows, int n, const uint4* __restrict__ src, uint4* dst,
                              int row_vec) {
  const size_t e = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= (size_t)n * row_vec) return;
  const size_t r = e / row_vec, c = e % row_vec;
  dst[e] = src[(size_t)rows[r] * row_vec + c];
}

}  // namespace
}  // namespace ta

using namespace ta;

extern "C" {

int tree_rope_fwd(const tree_plan_t* plan, const tree_bf16* q, const tree_bf16* k, tree_bf16* qr, tree_bf16* kr,
                  int Hq, int Hkv, int d, float theta, tree_stream_t stream) {
  int rc = plan_ok(plan);
  if (rc) return rc;
  if (!q || !k || !qr || !kr) return TREE_ERR_ARG;
  if ((d != 64 && d != 128) || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || !(theta > 0.f)) return TREE_ERR_SHAPE;
  for (const void* ptr : {(const void*)q, (const void*)k, (const void*)qr, (const void*)kr})
    if (reinterpret_cast<uintptr_t>(ptr) & 15) return TREE_ERR_ARG;
  rc = check_device();
  if (rc) return rc;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int N = plan->n_tokens;
  const int blocks = (N + kRopeTok - 1) / kRopeTok;
  if (d == 128)
    k_rope<128><<<blocks, kRopeThreads, 0, s>>>(plan->pos, N, theta, (const uint4*)q, (uint4*)qr, Hq,
                                                (const uint4*)k, (uint4*)kr, Hkv);
  else
    k_rope<64><<<blocks, kRopeThreads, 0, s>>>(plan->pos, N, theta, (const uint4*)q, (uint4*)qr, Hq,
                                               (const uint4*)k, (uint4*)kr, Hkv);
  return record_cuda(cudaGetLastError());
}

int tree_apply_weights(const tree_plan_t* plan, const tree_bf16* u, tree_bf16* dO, int H, int d,
                       tree_stream_t stream) {
  int rc = plan_ok(plan);
  if (rc) return rc;
  if (!u || !dO || !plan->w) return TREE_ERR_ARG;
  if (H <= 0 || d <= 0 || (H * d) % 8 != 0) return TREE_ERR_SHAPE;
  if ((reinterpret_cast<uintptr_t>(u) | reinterpret_cast<uintptr_t>(dO)) & 15) return TREE_ERR_ARG;
  rc = check_device();
  if (rc) return rc;
  const int per_token = H * d / 8;
  const size_t total = (size_t)plan->n_tokens * per_token;
  k_apply_weights<<<(unsigned)((total + 255) / 256), 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      plan->w, (const uint4*)u, (uint4*)dO, plan->n_tokens, per_token, per_token);
  return record_cuda(cudaGetLastError());
}

int tree_gather_rows(const int32_t* rows, int32_t n, const tree_bf16* src, tree_bf16* dst, int row_elems,
                     tree_stream_t stream) {
  if (!rows || !src || !dst || n <= 0) return TREE_ERR_ARG;
  if (row_elems <= 0 || row_elems % 8 != 0) return TREE_ERR_SHAPE;
  if ((reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst)) & 15) return TREE_ERR_ARG;
  int rc = check_device();
  if (rc) return rc;
  const int row_vec = row_elems / 8;
  const size_t total = (size_t)n * row_vec;
  k_gather_rows<<<(unsigned)((total + 255) / 256), 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      rows, n, reinterpret_cast<const uint4*>(src), reinterpret_cast<uint4*>(dst), row_vec);
  return record_cuda(cudaGetLastError());
}

}  // extern "C"
