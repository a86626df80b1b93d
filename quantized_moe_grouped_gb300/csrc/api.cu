// api.cu -- status strings and version of libqmoe.so.
#include "qmoe.h"

extern "C" const char* qmoe_status_string(qmoe_status_t st) {
    switch (st) {
        case QMOE_OK: return "ok";
        case QMOE_ERR_INVALID_ARG: return "invalid argument";
        case QMOE_ERR_UNSUPPORTED: return "unsupported shape or mode";
        case QMOE_ERR_CUDA: return "CUDA error (see cudaGetLastError)";
    }
    return "unknown status";
}

extern "C" int qmoe_version(void) { return 1; }
