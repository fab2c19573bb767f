// prefill.cu — placeholder until the tcgen05 kernel lands.
#include "pa_launch.h"
#include "../../include/pa.h"

namespace pa {
bool prefill_supported(int, int, int) { return false; }
int launch_prefill(const PrefillArgs&, const DeviceInfo&, cudaStream_t) { return PA_ERR_UNSUPPORTED; }
}  // namespace pa
