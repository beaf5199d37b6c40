// Test double of the CUDA runtime, for the host-policy tests of the expert cache on a
// machine without a GPU. It declares only what expert_cache.cu calls; harness.cpp defines
// the calls: copies are performed at once with memcpy and every call is appended to an
// operation log that the tests read back. Compiled only into the test harness, never into
// the library.
#pragma once

#include <stddef.h>

typedef struct FakeStream* cudaStream_t;
typedef struct FakeEvent* cudaEvent_t;

enum cudaError_t { cudaSuccess = 0, cudaErrorUnknown = 999 };
enum cudaMemcpyKind { cudaMemcpyHostToDevice = 1 };

#define cudaStreamNonBlocking 0x01
#define cudaEventDisableTiming 0x02

cudaError_t cudaStreamCreateWithFlags(cudaStream_t* stream, unsigned int flags);
cudaError_t cudaEventCreateWithFlags(cudaEvent_t* event, unsigned int flags);
cudaError_t cudaStreamSynchronize(cudaStream_t stream);
cudaError_t cudaStreamDestroy(cudaStream_t stream);
cudaError_t cudaEventDestroy(cudaEvent_t event);
cudaError_t cudaMemcpyAsync(void* dst, const void* src, size_t count, cudaMemcpyKind kind,
                            cudaStream_t stream);
cudaError_t cudaStreamWaitEvent(cudaStream_t stream, cudaEvent_t event, unsigned int flags);
cudaError_t cudaEventRecord(cudaEvent_t event, cudaStream_t stream);
