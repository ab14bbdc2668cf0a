// kernel_prefill_tc.cu -- tcgen05/TMEM prefill (placeholder until the kernel
// lands; the generic kernel serves every shape meanwhile).
#include "common.cuh"
#include "launch.h"

namespace attn {
bool prefill_tc_supported(const AttnParams &, int) { return false; }
int launch_prefill_tc(const AttnParams &, int, cudaStream_t) {
    set_error("tcgen05 prefill kernel not built");
    return 2;
}
}  // namespace attn
