// Library-wide entry points: version, status strings, device properties and
// the per-device error word the kernels raise bits in.
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
