// mxq_abi.cpp -- status strings and version of the C ABI declared in mxq.h.
#include "mxq.h"

extern "C" const char* mxq_status_string(int status) {
  switch (status) {
    case MXQ_OK: return "ok";
    case MXQ_EBADSHAPE:
      return "bad shape: sizes must be >= 0, within the limits and meet the method's multiples";
    case MXQ_EBADDTYPE: return "bad dtype: expected MXQ_F32 or MXQ_BF16";
    case MXQ_EBADOFFS: return "bad group offsets: G out of range, or offs/G inconsistent";
    case MXQ_EALIGN: return "misaligned pointer: buffers need 16-byte alignment (offs 4-byte)";
    case MXQ_EOVERLAP: return "overlapping buffers (or one past the top of memory)";
    case MXQ_ECUDA: return "CUDA runtime error at launch";
    case MXQ_ENULL: return "NULL pointer for a non-empty buffer";
    case MXQ_ESCRATCH:
      return "problem needs more scratch than the static area of the no-allocation call "
             "(M*N/32 > MXQ_NOALLOC_SCRATCH_BYTES)";
    default: return "unknown status";
  }
}

extern "C" int mxq_version(void) { return (1 << 16) | 0; }
