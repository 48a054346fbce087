// mla.cu -- MLA paged decode (latent form); see launch_mla.
#include "internal.h"
#include "sm103.cuh"

namespace fa {

int mla_chunk_tokens(int, int, int) { return 256; }

cudaError_t launch_mla(const MlaParams&, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace fa
