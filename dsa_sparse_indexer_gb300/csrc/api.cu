// Status strings and version of the DCP sparse-indexer C ABI.
#include "dsa.h"

extern "C" const char* dsa_status_string(dsa_status status) {
  switch (status) {
    case DSA_OK: return "ok";
    case DSA_ERR_INVALID_ARG: return "invalid argument";
    case DSA_ERR_UNSUPPORTED: return "unsupported configuration";
    case DSA_ERR_CUDA: return "CUDA launch error";
  }
  return "unknown status";
}

extern "C" int dsa_version(void) { return 100; }
