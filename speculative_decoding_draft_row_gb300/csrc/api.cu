// api.cu - status strings and version of the libtfd C ABI.
#include "common.cuh"

extern "C" const char* tfd_status_string(int status) {
  switch (status) {
    case TFD_OK: return "ok";
    case TFD_ERR_INVALID: return "invalid argument";
    case TFD_ERR_UNSUPPORTED: return "unsupported by this build";
    case TFD_ERR_WORKSPACE: return "workspace missing or too small";
    case TFD_ERR_CUDA: return "CUDA launch error";
    case TFD_ERR_DEVICE_DATA: return "bad ids, counts or positions in device data";
    case TFD_ERR_TIMEOUT: return "a bounded device wait gave up";
    default: return "unknown status";
  }
}

extern "C" int tfd_version(void) { return 100; }
