// Status strings and version of the libcconv.so C ABI (include/cconv.h).
#include "cconv.h"

extern "C" const char* cconv_status_string(int status) {
  switch (status) {
    case CCONV_OK:
      return "ok";
    case CCONV_ERR_INVALID:
      return "invalid argument (null pointer, size, stride or alignment out of range)";
    case CCONV_ERR_UNSUPPORTED:
      return "unsupported combination (no kernel for these sizes or this dtype)";
    case CCONV_ERR_LAUNCH:
      return "CUDA launch failed";
    case CCONV_ERR_TOO_LARGE:
      return "too much work for the fixed scratch of cca_qk_conv_noalloc (at most 2^30 units)";
    default:
      return "unknown status";
  }
}

extern "C" int cconv_abi_version(void) { return 6; }
