// mx_swap.h -- the block-scaled split GEMMs with swapped operands for
// decode-sized problems (csrc/gemm_mx_swap.cu).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace moe {

struct MxSwapArgs {
  const int* meta;           // meta[0] = number of row blocks
  const int* expert_of_rb;
  const int* counts;         // routed rows per expert
  const int* pad_offsets;    // padded segment starts: the routed rows of each row block
  const int* row_tok;
  const float* slot_w;
  void* act;                 // up: e4m3 [S_max, H] output
  void* act_sf;              // up: blocked scale tiles of act
  void* out;                 // down: bf16 [T, D] reduction target
  const void* sf_x;          // blocked scale tiles of the routed rows (xg or act)
  const void* sf_w;          // blocked scale tiles of the weights (W1 or W2)
  int* err;
  unsigned long long wait_limit_ns;
  int D, H;
  int n_col_tiles;           // 128-column tiles per row block (H / 128 up, D / 128 down)
  int k_blocks;              // K / 128
  int stall_test;            // test hook: the MMA issuer first waits on a barrier nothing arrives on
  int out_hint;              // 1: reductions into out carry an L2 evict_last hint
  float swiglu_limit;        // > 0: clamped SwiGLU
};

// map_w: the weights in boxes of 128 rows (e4m3 bytes, or packed E2M1 codes
// through a 16U4_ALIGN16B map when fp4w); map_x: the routed rows (xg up, act
// down) in boxes of 32 rows.
cudaError_t launch_up_mx_swap(const CUtensorMap& map_w1, const CUtensorMap& map_xg, const MxSwapArgs& args, int grid,
                              cudaStream_t stream, bool fp4w);
cudaError_t launch_down_mx_swap(const CUtensorMap& map_w2, const CUtensorMap& map_act, const MxSwapArgs& args,
                                int grid, cudaStream_t stream, bool pdl, bool fp4w);

}  // namespace moe
