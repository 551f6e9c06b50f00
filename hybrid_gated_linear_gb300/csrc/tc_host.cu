// tc_host.cu -- host side of the TMA path: the driver's tensor-map encoder, resolved once
// per process through the runtime's driver entry-point query, and the 3D bf16 maps the
// tensor-core kernels read and write.
#include <mutex>

#include "lizard_internal.h"

namespace lz {

namespace {
using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                 const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                 const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                 CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled get_encode() {
  static EncodeTiled fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiled>(ptr);
  });
  return fn;
}
}  // namespace

int ctas_per_wave(int per_sm) {
  static std::mutex mu;
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148 * per_sm;
  std::lock_guard<std::mutex> lock(mu);
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
    cache[dev] = n;
  }
  return cache[dev] * per_sm;
}

std::mutex& side_stream_lock() {
  static std::mutex mu;
  return mu;
}

SideStream* side_stream() {
  static SideStream per_dev[64];
  static bool ready[64] = {false};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  if (!ready[dev]) {
    SideStream& s = per_dev[dev];
    if (cudaStreamCreateWithFlags(&s.stream, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&s.fork, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&s.join, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&s.done, cudaEventDisableTiming) != cudaSuccess)
      return nullptr;
    ready[dev] = true;
  }
  return &per_dev[dev];
}

bool tma_encode_available() { return get_encode() != nullptr; }

namespace {
bool make_map(CUtensorMap* m, CUtensorMapDataType dt, uint32_t esize, const void* base,
              uint64_t dim0, uint64_t dim1, uint64_t dim2, uint32_t box0, uint32_t box1,
              CUtensorMapSwizzle sw) {
  EncodeTiled enc = get_encode();
  if (!enc) return false;
  cuuint64_t dims[3] = {dim0, dim1, dim2};
  cuuint64_t strides[2] = {dim0 * esize, dim0 * dim1 * esize};
  cuuint32_t box[3] = {box0, box1, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, dt, 3, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
}  // namespace

bool make_tma_map_f32(CUtensorMap* m, const void* base, uint64_t dim0, uint64_t dim1,
                      uint64_t dim2, uint32_t box0, uint32_t box1, CUtensorMapSwizzle sw) {
  return make_map(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, base, dim0, dim1, dim2, box0, box1, sw);
}

bool make_tma_map_bf16(CUtensorMap* m, const void* base, uint64_t dim0, uint64_t dim1,
                       uint64_t dim2, uint32_t box0, uint32_t box1, CUtensorMapSwizzle sw) {
  return make_map(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dim0, dim1, dim2, box0, box1, sw);
}

}  // namespace lz
