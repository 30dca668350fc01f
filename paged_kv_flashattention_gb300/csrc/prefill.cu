// Varlen prefill / extend attention (tcgen05 + TMEM).  Placeholder.
#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

PA_ERROR_WORD_ACCESSOR(error_word_prefill)

cudaError_t launch_prefill(const pa_prefill_params &, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace pa
