// prefill.cu -- placeholder until the tcgen05 prefill kernel lands.
#include "internal.h"
namespace gqa {
bool prefill_supported(int) { return false; }
cudaError_t prefill_launch(const PrefillArgs&, int, cudaStream_t) { return cudaErrorNotSupported; }
}  // namespace gqa
