// attn_params.h -- launch parameters shared by the decode-attention kernels
// (attn.cu: the register-direct kernels and the split combine; attn_tc.cu: the
// tensor-memory verification kernel) and their host launchers.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.h"

namespace lynx {

// Shared-window address of the first byte of dynamic shared memory for a
// kernel without static shared memory: the block's reserved shared memory
// (1 KiB on sm_100-class GPUs) comes first.  The host checks the device
// attribute before launching and the kernels check the address themselves
// (their table loads use it as an immediate offset).
constexpr uint32_t kSmemBase = 1024;

struct AttnParams {
  const uint16_t* q;
  const uint8_t *ka, *kr, *va, *vr;
  const float *km, *vm;
  const uint16_t *kt, *vt;  // draft tokens' own keys / values, or null
  const int32_t* bt;        // block table [batch][NB] of physical pages, or null (dense)
  int64_t nphys;            // physical pages behind the table
  float* part;
  float* out;
  int batch, T, Hq, Hkv, G, R, nrg;
  int64_t L, NB, NCH;
  int64_t n_chunks;  // units x NCH: the flattened (unit, chunk) space
  int n_cta;         // CTAs of the attention grid
  int P, C, NC, lgP, lgC;
  float scale_log2;
};

// The split combine over the partials (m, l, o) of RP query rows per unit,
// launched as a programmatic dependent of the attention grid (attn.cu).
cudaError_t launch_attn_combine(const AttnParams& prm, int RP, cudaStream_t stream);

// The verification pass on the tensor-memory path (attn_tc.cu): full codes,
// 32 query rows per pass, tiles of 128 tokens.  prm.NCH, prm.n_chunks and
// prm.n_cta count tiles; attn_tc_ctas gives the grid.
int attn_tc_ctas(int batch, int Hkv, int nrg, int64_t ntiles, int sms);
cudaError_t launch_attn_tc(const AttnParams& prm, const ExpandTable& tab, cudaStream_t stream);
cudaError_t read_attn_tc_flags(unsigned int* flag);

}  // namespace lynx
