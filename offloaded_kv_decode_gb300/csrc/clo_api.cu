// clo_api.cu -- status helpers of the libclo C ABI (host only).
#include "clo.h"

extern "C" const char* clo_status_string(clo_status s) {
    switch (s) {
        case CLO_OK: return "CLO_OK";
        case CLO_ERR_INVALID_ARG: return "CLO_ERR_INVALID_ARG";
        case CLO_ERR_UNSUPPORTED: return "CLO_ERR_UNSUPPORTED";
        case CLO_ERR_CUDA: return "CLO_ERR_CUDA";
        case CLO_ERR_BAD_INDEX: return "CLO_ERR_BAD_INDEX";
        case CLO_ERR_WORKSPACE: return "CLO_ERR_WORKSPACE";
        case CLO_ERR_TIMEOUT: return "CLO_ERR_TIMEOUT";
    }
    return "CLO_ERR_UNKNOWN";
}

extern "C" int clo_version(void) { return 10300; }  // 1.3.0

extern "C" clo_status clo_check_error_flag(int32_t host_err_flag) {
    if (host_err_flag == 0) return CLO_OK;
    return (host_err_flag & CLO_FLAG_TIMEOUT) ? CLO_ERR_TIMEOUT : CLO_ERR_BAD_INDEX;
}
