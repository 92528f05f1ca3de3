// Back-transformation of the recorded reflectors (bb_vectors.cu).
#pragma once

#include <cuda_runtime.h>

namespace bb {

// U = L_1 L_2 ... and V = R_1 R_2 ... (column-major, n x n, leading
// dimensions ldu, ldv; either may be null) from the reflector record of a
// whole reduction of bandwidth bw with tile width tw: reflector index
// 2 (steps before this one in the pass order) + side, v at rec_v[index *
// stride ..], tau at rec_tau[index].  One launch per sweep and matrix.
template <typename T>
cudaError_t run_back_transform(long long n, int bw, int tw, const T* rec_v, const T* rec_tau, int stride, T* U,
                               long long ldu, T* V, long long ldv, int num_sms, cudaStream_t s, long long* launches);

}  // namespace bb
