// Host-side entry points of the chunkwise prefill, one per variant (each
// instantiated in its own translation unit so they compile in parallel).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "kernels.h"

namespace la {
namespace chunk {

struct Maps {
    CUtensorMap q, k, v, g, o;
};

struct Params;

cudaError_t launch_norm(int dk, int dv, const Maps& m, const Params& p, int BH, cudaStream_t s);
cudaError_t launch_gla(int dk, int dv, const Maps& m, const Params& p, int BH, cudaStream_t s);
cudaError_t launch_gdn(int dk, int dv, const Maps& m, const Params& p, int BH, cudaStream_t s);

}  // namespace chunk
}  // namespace la
