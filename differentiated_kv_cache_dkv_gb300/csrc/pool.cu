// pool.cu -- pool reset (k_init_pool) and page dequantisation (k_dequant).
//
// DiffKV (arXiv 2412.03131), Pith review, "Core claim": a GPU-resident
// manager with unified pages, a circular free page list and a bidirectional
// page table.  A fresh pool lists every page as free in id order.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "dkv_internal.cuh"

namespace dkv {

namespace {

constexpr int kInitThreads = 256;
constexpr int kDequantThreads = 256;

__global__ void __launch_bounds__(kInitThreads) k_init_pool(dkv_pool p) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < p.F; i += stride) {
    p.free_list[i] = static_cast<int32_t>(i);
    p.rev_unit[i] = -1;
    p.rev_idx[i] = -1;
    p.page_cls[i] = 0;
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    p.cursors[0] = 0;
    p.cursors[1] = static_cast<uint64_t>(p.F);
    *p.status = 0;
  }
}

// One block per page.  x' = fma(q, scale, zero) in fp32, no second rounding.
__global__ void __launch_bounds__(kDequantThreads) k_dequant(dkv_pool p, const int32_t *ids, int32_t one_id,
                                                             float *k_out, float *v_out, int32_t *pos_out) {
  const int64_t b = blockIdx.x;
  const int32_t id = ids ? ids[b] : one_id;
  const int64_t P = p.P;
  const PageGeom g = page_geom(p.scheme, p.P);
  const int cls = (id >= 0 && id < p.F) ? p.page_cls[id] : 0;
  const uint8_t *pg = p.pages + static_cast<int64_t>(id >= 0 && id < p.F ? id : 0) * g.bytes;
  float *ko = k_out + b * 2 * P * 128;
  float *vo = v_out + b * 2 * P * 128;
  for (int64_t e = threadIdx.x; e < 2 * P * 128; e += blockDim.x) {
    const int64_t s = e >> 7;
    const int d = static_cast<int>(e & 127);
    const bool high = cls == DKV_CLASS_K8V4;
    const bool exists = cls == DKV_CLASS_K4V2 || (high && s < P);
    float kx = 0.0f, vx = 0.0f;
    int32_t pos = -1;
    if (exists) {
      // channel d of a slot at width w: bits [w (d mod 8/w), ...) of byte d w / 8
      const int kw = high ? g.kh : g.kh >> 1, vw = high ? g.vh : g.vh >> 1;
      const uint32_t qk = (pg[s * 16 * kw + (d * kw >> 3)] >> ((d * kw) & 7)) & ((1u << kw) - 1u);
      const uint32_t qv = (pg[g.vbase + s * 16 * vw + (d * vw >> 3)] >> ((d * vw) & 7)) & ((1u << vw) - 1u);
      const __half *meta = reinterpret_cast<const __half *>(pg + g.meta + 8 * s);
      kx = __fmaf_rn(static_cast<float>(qk), __half2float(meta[0]), __half2float(meta[1]));
      vx = __fmaf_rn(static_cast<float>(qv), __half2float(meta[2]), __half2float(meta[3]));
      pos = *reinterpret_cast<const int32_t *>(pg + g.pos + 4 * s);
    }
    ko[e] = kx;
    vo[e] = vx;
    if (d == 0) pos_out[b * 2 * P + s] = pos;
  }
}

}  // namespace

cudaError_t launch_init_pool(const dkv_pool &p, cudaStream_t s) {
  int64_t blocks = (p.F + kInitThreads - 1) / kInitThreads;
  if (blocks > 4096) blocks = 4096;
  if (blocks < 1) blocks = 1;
  k_init_pool<<<static_cast<int>(blocks), kInitThreads, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_dequant(const dkv_pool &p, const int32_t *ids, int32_t one_id, int32_t n, float *k_out,
                           float *v_out, int32_t *pos_out, cudaStream_t s) {
  k_dequant<<<n, kDequantThreads, 0, s>>>(p, ids, one_id, k_out, v_out, pos_out);
  return cudaGetLastError();
}

}  // namespace dkv
