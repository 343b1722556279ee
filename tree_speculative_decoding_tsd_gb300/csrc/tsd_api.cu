// Library-wide C entry points: status text and version.
#include "tsd.h"

extern "C" const char* tsd_status_string(tsd_status s) {
  switch (s) {
    case TSD_OK: return "ok";
    case TSD_ERR_INVALID_ARG: return "invalid argument (size, null or misaligned pointer, short workspace)";
    case TSD_ERR_UNSUPPORTED: return "unsupported configuration";
    case TSD_ERR_CUDA: return "CUDA runtime or launch error";
    case TSD_ERR_DEVICE: return "device-side error (see the err word)";
    case TSD_ERR_DEVICE_TIMEOUT: return "a bounded device wait gave up";
  }
  return "unknown status";
}

extern "C" int tsd_version(void) { return 100; }
