// tensormap.cu -- host helpers: TMA descriptor encoding (driver entry point looked up through the
// runtime, so the library does not link libcuda directly) and cached device properties.
#include <atomic>
#include <mutex>

#include "internal.h"

namespace wql {
namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess) {
      fn = reinterpret_cast<EncodeTiledFn>(p);
    }
  });
  return fn;
}

}  // namespace

bool make_tmap_2d(CUtensorMap* map, CUtensorMapDataType dtype, int elem_bytes, const void* base, uint64_t inner,
                  uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer,
                  CUtensorMapSwizzle swizzle, std::string* err) {
  EncodeTiledFn enc = get_encode();
  if (!enc) {
    if (err) *err = "cuTensorMapEncodeTiled is not available from the driver";
    return false;
  }
  (void)elem_bytes;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, dtype, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    if (err)
      *err = "cuTensorMapEncodeTiled failed (code " + std::to_string((int)r) + ") for a " + std::to_string(outer) +
             "x" + std::to_string(inner) + " tensor with box " + std::to_string(box_outer) + "x" +
             std::to_string(box_inner);
    return false;
  }
  return true;
}

bool make_tmap_3d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, uint64_t d0, uint64_t d1,
                  uint64_t d2, uint64_t stride1, uint64_t stride2, uint32_t b0, uint32_t b1, uint32_t b2,
                  CUtensorMapSwizzle swizzle, std::string* err) {
  EncodeTiledFn enc = get_encode();
  if (!enc) {
    if (err) *err = "cuTensorMapEncodeTiled is not available from the driver";
    return false;
  }
  const cuuint64_t dims[3] = {d0, d1, d2};
  const cuuint64_t strides[2] = {stride1, stride2};
  const cuuint32_t box[3] = {b0, b1, b2};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, dtype, 3, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    if (err) *err = "cuTensorMapEncodeTiled (3D) failed (code " + std::to_string((int)r) + ")";
    return false;
  }
  return true;
}

int num_sms() {
  static std::atomic<int> cache[64];  // racing first calls store the same count
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return 148;
  int n = cache[dev].load(std::memory_order_relaxed);
  if (n == 0) {
    int v = 0;
    cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    n = v > 0 ? v : 148;
    cache[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

int pick_k_split(const void* kernel, int threads, int smem_bytes, int units, int kblocks, bool pow2, bool balanced) {
  struct Entry {
    const void* k;
    int dev, smem, cap[9];
  };
  static std::mutex mu;
  static Entry cache[32];
  static int n_cache = 0;
  int dev = 0;
  cudaGetDevice(&dev);
  int cap[9] = {0};
  {
    std::lock_guard<std::mutex> lock(mu);
    int found = -1;
    for (int i = 0; i < n_cache; ++i)
      if (cache[i].k == kernel && cache[i].dev == dev && cache[i].smem == smem_bytes) found = i;
    if (found < 0) {
      Entry e{kernel, dev, smem_bytes, {0}};
      for (int S = 1; S <= 8; ++S) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(1, S, 1);
        cfg.blockDim = dim3(threads, 1, 1);
        cfg.dynamicSmemBytes = smem_bytes;
        cudaLaunchAttribute attr;
        attr.id = cudaLaunchAttributeClusterDimension;
        attr.val.clusterDim.x = 1;
        attr.val.clusterDim.y = S;
        attr.val.clusterDim.z = 1;
        cfg.attrs = &attr;
        cfg.numAttrs = 1;
        int clusters = 0;
        if (cudaOccupancyMaxActiveClusters(&clusters, kernel, &cfg) != cudaSuccess) {
          cudaGetLastError();
          clusters = 0;
        }
        e.cap[S] = clusters * S;
      }
      if (n_cache < 32) cache[n_cache++] = e;
      for (int S = 0; S <= 8; ++S) cap[S] = e.cap[S];
    } else {
      for (int S = 0; S <= 8; ++S) cap[S] = cache[found].cap[S];
    }
  }
  const int sms = num_sms();
  if (balanced) {
    // Weight streaming is bound by each SM's copy rate, so the time is set by the busiest SM: the
    // co-resident CTAs of an SM share it.  Model: rounds = ceil(CTAs / co-resident capacity); an SM
    // runs ceil(CTAs in a round / SMs) CTAs of kblocks / S blocks each, plus a fixed cost per CTA
    // (launch, activation fetch, reduction) of about kFixed blocks.  Smallest cost wins; ties go
    // to the smaller S, which also leaves room on the SMs for the next layer's early start.
    constexpr double kFixed = 4.0;
    int best = 1;
    double best_cost = 1e30;
    for (int S = 1; S <= 8 && S <= (kblocks > 0 ? kblocks : 1); ++S) {
      if (pow2 && (S & (S - 1))) continue;
      if (cap[S] <= 0) continue;
      const long long ctas = (long long)units * S;
      const long long rounds = (ctas + cap[S] - 1) / cap[S];
      const long long per_round = ctas < cap[S] ? ctas : cap[S];
      const long long per_sm = (per_round + sms - 1) / sms;
      const double cost = (double)(rounds * per_sm) * ((double)((kblocks + S - 1) / S) + kFixed);
      if (cost < best_cost - 1e-9) {
        best_cost = cost;
        best = S;
      }
    }
    return best;
  }
  // About one CTA per SM: a decode layer then leaves room on every SM for the next layer's CTAs,
  // which start streaming their weights early (programmatic dependent launch).
  int S = sms / (units > 0 ? units : 1);
  if (S > 8) S = 8;
  if (S > kblocks) S = kblocks;
  if (S < 1) S = 1;
  if (pow2)
    while (S & (S - 1)) S &= S - 1;
  while (S > 1 && units * S > cap[S]) S = pow2 ? S / 2 : S - 1;
  return S;
}

}  // namespace wql
