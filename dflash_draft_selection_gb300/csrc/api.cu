// api.cu -- status strings and the device error word of the DFlash 2 library.
#include "host.hpp"

namespace dfl {
unsigned int read_error_topk(bool clear);
unsigned int read_error_verify(bool clear);
unsigned int read_error_gate(bool clear);
}  // namespace dfl

extern "C" const char *dflash2_status_string(dflash2_status s) {
    switch (s) {
        case DFLASH2_OK: return "ok";
        case DFLASH2_ERR_INVALID_ARG: return "invalid argument";
        case DFLASH2_ERR_UNSUPPORTED: return "unsupported";
        case DFLASH2_ERR_CUDA: return "CUDA error";
        case DFLASH2_ERR_WORKSPACE: return "workspace too small";
    }
    return "unknown status";
}

extern "C" dflash2_status dflash2_device_error(uint32_t *code, int clear) {
    if (!code) return DFLASH2_ERR_INVALID_ARG;
    if (cudaDeviceSynchronize() != cudaSuccess) return DFLASH2_ERR_CUDA;
    *code = dfl::read_error_topk(clear != 0) | dfl::read_error_verify(clear != 0) |
            dfl::read_error_gate(clear != 0);
    return cudaPeekAtLastError() == cudaSuccess ? DFLASH2_OK : DFLASH2_ERR_CUDA;
}
