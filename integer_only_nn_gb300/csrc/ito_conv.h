// Host launchers of the conv / pooling kernels (ito_conv.cu).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace ito {

// 3x3, pad 1: P[(b,oh,ow)][(kh,kw,ic)] = bf16(x[b][oh*s-1+kh][ow*s-1+kw][ic]) (0 in the padding)
int launch_im2col(const int8_t* x, int B, int H, int W, int IC, int OH, int OW, int stride, uint16_t* P, int64_t ldp,
                  cudaStream_t s);
// D[b][ih][iw][ic] = sum of the patch entries taken from (ih, iw); atomicMax(d_max, max |D|)
int launch_col2im(const int32_t* Dcol, int B, int H, int W, int IC, int OH, int OW, int stride, int32_t* D,
                  uint32_t* d_max, cudaStream_t s);
int launch_gap_fwd(const int8_t* A, int B, int HW, int C, int32_t* P, uint32_t* d_max, cudaStream_t s);
int launch_gap_bwd(const int8_t* dP, const int8_t* A, int B, int HW, int C, int8_t* E, uint16_t* Eb, cudaStream_t s);

}  // namespace ito
