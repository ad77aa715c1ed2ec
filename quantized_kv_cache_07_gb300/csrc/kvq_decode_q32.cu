// Decode kernels with the two-part fp16 query (q_bits 32: fp16 high part in
// registers, fp16 low part from shared memory, one more MMA per k-slice) for
// every code format, symmetric and asymmetric.  The kernel template lives in
// kvq_decode_impl.cuh.
#include "kvq_decode_impl.cuh"

namespace kvq {

int decode_ctas_per_sm_q32(int k_bits, int v_bits, bool asym, int B, bool rows) {
  if (asym) {
    if (k_bits == 8 && v_bits == 8) return Kernel<8, 8, true, true>::ctas_per_sm(B, rows);
    if (k_bits == 4 && v_bits == 4) return Kernel<4, 4, true, true>::ctas_per_sm(B, rows);
    if (k_bits == 4 && v_bits == 8) return Kernel<4, 8, true, true>::ctas_per_sm(B, rows);
    if (k_bits == 8 && v_bits == 4) return Kernel<8, 4, true, true>::ctas_per_sm(B, rows);
    if (k_bits == 2 && v_bits == 2) return Kernel<2, 2, true, true>::ctas_per_sm(B, rows);
    return 0;
  }
  if (k_bits == 8 && v_bits == 8) return Kernel<8, 8, false, true>::ctas_per_sm(B, rows);
  if (k_bits == 4 && v_bits == 4) return Kernel<4, 4, false, true>::ctas_per_sm(B, rows);
  if (k_bits == 4 && v_bits == 8) return Kernel<4, 8, false, true>::ctas_per_sm(B, rows);
  if (k_bits == 8 && v_bits == 4) return Kernel<8, 4, false, true>::ctas_per_sm(B, rows);
  if (k_bits == 2 && v_bits == 2) return Kernel<2, 2, false, true>::ctas_per_sm(B, rows);
  return 0;
}

cudaError_t launch_decode_q32(const DecodeArgs& a, cudaStream_t s) {
  const int kb = a.c.k_bits, vb = a.c.v_bits;
  if (a.c.asym) {
    if (kb == 8 && vb == 8) return Kernel<8, 8, true, true>::launch(a, s);
    if (kb == 4 && vb == 4) return Kernel<4, 4, true, true>::launch(a, s);
    if (kb == 4 && vb == 8) return Kernel<4, 8, true, true>::launch(a, s);
    if (kb == 8 && vb == 4) return Kernel<8, 4, true, true>::launch(a, s);
    if (kb == 2 && vb == 2) return Kernel<2, 2, true, true>::launch(a, s);
    return cudaErrorInvalidValue;
  }
  if (kb == 8 && vb == 8) return Kernel<8, 8, false, true>::launch(a, s);
  if (kb == 4 && vb == 4) return Kernel<4, 4, false, true>::launch(a, s);
  if (kb == 4 && vb == 8) return Kernel<4, 8, false, true>::launch(a, s);
  if (kb == 8 && vb == 4) return Kernel<8, 4, false, true>::launch(a, s);
  if (kb == 2 && vb == 2) return Kernel<2, 2, false, true>::launch(a, s);
  return cudaErrorInvalidValue;
}

}  // namespace kvq
