// Host-side declarations every translation unit of liblayer_rnn.so shares:
// the launch counter and the TMA map encoder.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

namespace lr {

// kernels launched by this library (all handles, all threads); the phase
// timing of a handle reports its share per phase
extern std::atomic<int64_t> g_kernel_launches;

// encode a tiled TMA map (bf16 / fp32, rank 2 or 3, 128-byte swizzle)
bool tma_encode(void* map, int rank, bool bf, const void* ptr, const uint64_t* dims,
                const uint64_t* strides_bytes, const uint32_t* box);

}  // namespace lr
