// Tensor-core (tcgen05/TMEM) chunked forward for bf16 I/O.
// Placeholder until the tcgen05 kernel lands: routes to the CUDA-core path.
#include "kda_internal.cuh"

namespace kda {
cudaError_t launch_chunk_fwd_tc(const ChunkFwdArgs& a) { return launch_chunk_fwd_simt(a, KDA_BF16); }
}  // namespace kda
