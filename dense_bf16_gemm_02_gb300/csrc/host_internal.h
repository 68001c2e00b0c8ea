// Host-side services the GEMM translation unit (hk_gemm.cu) provides to the
// other entry points of the library: the thread-local error string, the
// per-device status word of the one-shot entry points, the device check,
// the tensor-map encoder and process-unique launch ids.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cstdint>

#include "../../include/hk_gemm.h"

namespace hk_host {

// Records `msg` as the calling thread's last error and returns `s`.
hk_status set_error(hk_status s, const char* msg);

// The device status word ([0] error bits, [1] aborted launch id) shared by
// every one-shot entry point on `device`; allocated on first use.
hk_status status_word(int device, uint32_t** out);

// HK_OK when `device` is a compute capability 10.3 device (sets the error
// string otherwise); `sm_count` receives its number of SMs.
hk_status check_device(int device, int* sm_count);

// cuTensorMapEncodeTiled from the driver.
hk_status tensor_map_encoder(PFN_cuTensorMapEncodeTiled_v12000* out);

uint32_t next_launch_id();

}  // namespace hk_host
