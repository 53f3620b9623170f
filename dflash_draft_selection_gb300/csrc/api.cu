// api.cu -- status strings and the device error word of the DFlash 2 library.
#include "host.hpp"

#include <mutex>

namespace dfl {
unsigned int read_error_topk(bool clear);
unsigned int read_error_verify(bool clear);
unsigned int read_error_gate(bool clear);
unsigned int read_error_lmhead(bool clear);

// dflash2_test_hold's setting: read by every scan launch (make_geom).
static std::mutex g_hold_mu;
static const unsigned int *g_hold_flag = nullptr;
static long long g_hold_cycles = 0;

void scan_hold(const unsigned int **flag, long long *cycles) {
    std::lock_guard<std::mutex> lock(g_hold_mu);
    *flag = g_hold_flag;
    *cycles = g_hold_cycles;
}
}  // namespace dfl

extern "C" dflash2_status dflash2_test_hold(const uint32_t *flag, int64_t max_cycles) {
    if (flag && (max_cycles < 1 || max_cycles > (int64_t(1) << 32) ||
                 (reinterpret_cast<uintptr_t>(flag) & 3) != 0))
        return DFLASH2_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(dfl::g_hold_mu);
    dfl::g_hold_flag = flag;
    dfl::g_hold_cycles = flag ? max_cycles : 0;
    return DFLASH2_OK;
}

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
            dfl::read_error_gate(clear != 0) | dfl::read_error_lmhead(clear != 0);
    return cudaPeekAtLastError() == cudaSuccess ? DFLASH2_OK : DFLASH2_ERR_CUDA;
}
