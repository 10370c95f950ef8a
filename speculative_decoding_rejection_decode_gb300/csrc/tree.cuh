// Token-tree verification (tree.cu): arguments and launcher, shared with the
// entry point in specdec.cu.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace specdec {

constexpr int kTreeMaxChildren = 256;  // candidates tested per node; more set the capacity bit

struct TreeArgs {
  const void* logits;        // [N, V] float or bf16: target row of every node
  const float* q;            // [N, V] draft row of every node (rows of nodes with children are read); null at T == 0
  const int32_t* tok;        // [N] token of every node (node 0 of a request: unused)
  const int32_t* par;        // [N] parent within the request (node 0: -1)
  const int32_t* cu;         // [B+1] node offsets of the requests
  int B;
  int V;
  float c;                   // log2(e) / T, 0 for greedy
  uint64_t seed;
  uint64_t req_offset;       // generator request index = req_offset + b
  int32_t* out_tokens;       // [N]
  int32_t* out_nacc;         // [B]
  int32_t* out_path;         // [N] or null
  uint32_t* err;             // sticky device error word
  unsigned long long* counter;  // request counter (zeroed by the launcher)
  int vec_ok;                // rows are 16-byte aligned
};

// Queues the walk of every request on st (num_sms: multiprocessor count).
// Returns SPECDEC_OK or SPECDEC_ERR_CUDA.
int launch_tree(const TreeArgs& a, int dtype, int num_sms, cudaStream_t st);

}  // namespace specdec
