// Library-wide entry points: version, status strings, device properties and
// the per-device error word the kernels raise bits in.
#include <cuda.h>

#include <mutex>

#include "common.cuh"

namespace {

// One error word per device; kernels receive its address as an argument.
__device__ unsigned int g_pkv_error_word;

constexpr int kMaxDevices = 64;

struct DeviceSlot {
  bool ready = false;
  pkv::DeviceInfo info{};
  unsigned int* error_word = nullptr;
};

std::mutex g_mutex;
DeviceSlot g_slots[kMaxDevices];

int prepare_slot(DeviceSlot** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PKV_ECUDA;
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceSlot& s = g_slots[dev];
  if (!s.ready) {
    if (cudaDeviceGetAttribute(&s.info.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return PKV_ECUDA;
    if (cudaDeviceGetAttribute(&s.info.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
      return PKV_ECUDA;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_pkv_error_word) != cudaSuccess) return PKV_ECUDA;
    s.error_word = static_cast<unsigned int*>(p);
    s.ready = true;
  }
  *out = &s;
  return PKV_OK;
}

}  // namespace

namespace pkv {

int device_info(DeviceInfo* info) {
  DeviceSlot* s = nullptr;
  int st = prepare_slot(&s);
  if (st != PKV_OK) return st;
  *info = s->info;
  return PKV_OK;
}

unsigned int* device_error_word(int* status) {
  DeviceSlot* s = nullptr;
  *status = prepare_slot(&s);
  return *status == PKV_OK ? s->error_word : nullptr;
}

namespace {
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
std::once_flag g_encode_once;
EncodeTiledFn g_encode = nullptr;
}  // namespace

int encode_bf16_3d(void* map, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint32_t b0, uint32_t b1,
                   uint32_t b2) {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  });
  if (!g_encode) return PKV_ECUDA;
  const cuuint64_t dims[3] = {d0, d1, d2};
  const cuuint64_t strides[2] = {d0 * 2, d0 * d1 * 2};
  const cuuint32_t box[3] = {b0, b1, b2};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = g_encode(static_cast<CUtensorMap*>(map), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                              const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? PKV_OK : PKV_ECUDA;
}

int encode_paged_kv(void* map, const void* base, uint32_t block_size, uint32_t hkv, uint64_t num_blocks,
                    int elem_bytes) {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  });
  if (!g_encode || (elem_bytes != 1 && elem_bytes != 2)) return PKV_ECUDA;
  // dims innermost first: head_dim, token in block, KV head, block; the
  // token stride (all heads of a token) is larger than the head stride
  const cuuint64_t row = 128 * static_cast<cuuint64_t>(elem_bytes);
  const cuuint64_t dims[4] = {128, block_size, hkv, num_blocks};
  const cuuint64_t strides[3] = {hkv * row, row, static_cast<cuuint64_t>(block_size) * hkv * row};
  const cuuint32_t box[4] = {128u / static_cast<cuuint32_t>(elem_bytes), 16, hkv, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUtensorMapDataType type = elem_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  const CUresult r = g_encode(static_cast<CUtensorMap*>(map), type, 4, const_cast<void*>(base), dims, strides, box,
                              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? PKV_OK : PKV_ECUDA;
}

}  // namespace pkv

extern "C" int pkv_version(void) { return 10000; }

extern "C" const char* pkv_status_string(int status) {
  switch (status) {
    case PKV_OK: return "ok";
    case PKV_EINVAL: return "invalid argument";
    case PKV_EUNSUPPORTED: return "unsupported shape or dtype";
    case PKV_EALIGN: return "pointer not 16-byte aligned";
    case PKV_ECUDA: return "CUDA runtime error";
    case PKV_EWORKSPACE: return "workspace missing or too small";
    case PKV_ESCRATCH: return "sizes need more split scratch than the no-allocation entry point holds";
    default: return "unknown status";
  }
}

extern "C" int pkv_get_device_error(uint32_t* flags, int reset) {
  if (!flags) return PKV_EINVAL;
  int st = PKV_OK;
  unsigned int* word = pkv::device_error_word(&st);
  if (st != PKV_OK) return st;
  if (cudaDeviceSynchronize() != cudaSuccess) return PKV_ECUDA;
  unsigned int v = 0;
  if (cudaMemcpy(&v, word, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return PKV_ECUDA;
  *flags = v;
  if (reset) {
    const unsigned int zero = 0;
    if (cudaMemcpy(word, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) return PKV_ECUDA;
  }
  return PKV_OK;
}
