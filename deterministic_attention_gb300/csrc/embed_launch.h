// Internal interface of the embedding-gradient kernels (embed_grad.cu): the
// argument block and the launch function.  Not part of the public API.
#pragma once
#include <cuda_runtime.h>

namespace detattn {

struct EmbedArgs {
  const int* ids;      // int32 [N] token ids
  const void* dy;      // bf16 [N, E]
  float* dw;           // fp32 [V, E]
  int N, V, E;
  // Workspace (caller-owned; see embed_grad_workspace_bytes in detattn.h).
  int* counts;         // [V]      tokens per id
  int* offsets;        // [V + 1]  exclusive prefix of counts
  int* cursor;         // [V]      slots handed out per id
  int* unsorted;       // [N]      tokens grouped by id, any order within an id
  int* sorted;         // [N]      tokens grouped by id, ascending within an id
  float* head;         // [ceil(N / 32), E] partial rows of ids that began in an earlier run
  float* tail;         // [ceil(N / 32), E] partial rows of ids that go on past their run
};

// Queues the whole gradient on `st` (one memset and up to six kernels).
cudaError_t launch_embed_grad(const EmbedArgs& a, int sms, cudaStream_t st);
// Number of kernels launch_embed_grad queues for N tokens.
int embed_grad_launches(int N);
// Read-and-clear of the embedding step's device status word (bit 0: an id
// outside [0, V) was skipped); synchronous on `st`.
cudaError_t take_embed_status(cudaStream_t st, unsigned* out);

}  // namespace detattn
