#include "gdn_internal.h"
namespace gdn {
cudaError_t launch_chunked(const ChunkedParams &, cudaStream_t, int) { return cudaErrorNotSupported; }
}
