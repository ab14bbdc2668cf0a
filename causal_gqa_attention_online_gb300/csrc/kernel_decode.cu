// kernel_decode.cu -- split-KV tensor-core decode (placeholder until the
// kernel lands; the generic kernel serves every shape meanwhile).
#include "common.cuh"
#include "launch.h"

namespace attn {
bool decode_supported(const AttnParams &, int) { return false; }
int decode_split_len(const AttnParams &p, int) { return p.K > 0 ? p.K : 1; }
int launch_decode(const AttnParams &, int, cudaStream_t) {
    set_error("decode kernel not built");
    return 2;
}
}  // namespace attn
