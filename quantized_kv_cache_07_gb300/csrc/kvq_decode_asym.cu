// Decode kernels for the asymmetric formats (per-token scale and zero point on
// both K and V) with the fp16 or int8 query.  The kernel template lives in
// kvq_decode_impl.cuh.
#include "kvq_decode_impl.cuh"

namespace kvq {

int decode_ctas_per_sm_asym(int k_bits, int v_bits, int B, bool rows) {
  if (k_bits == 8 && v_bits == 8) return Kernel<8, 8, true, false>::ctas_per_sm(B, rows);
  if (k_bits == 4 && v_bits == 4) return Kernel<4, 4, true, false>::ctas_per_sm(B, rows);
  if (k_bits == 4 && v_bits == 8) return Kernel<4, 8, true, false>::ctas_per_sm(B, rows);
  if (k_bits == 8 && v_bits == 4) return Kernel<8, 4, true, false>::ctas_per_sm(B, rows);
  if (k_bits == 2 && v_bits == 2) return Kernel<2, 2, true, false>::ctas_per_sm(B, rows);
  return 0;
}

cudaError_t launch_decode_asym(const DecodeArgs& a, cudaStream_t s) {
  const int kb = a.c.k_bits, vb = a.c.v_bits;
  if (kb == 8 && vb == 8) return Kernel<8, 8, true, false>::launch(a, s);
  if (kb == 4 && vb == 4) return Kernel<4, 4, true, false>::launch(a, s);
  if (kb == 4 && vb == 8) return Kernel<4, 8, true, false>::launch(a, s);
  if (kb == 8 && vb == 4) return Kernel<8, 4, true, false>::launch(a, s);
  if (kb == 2 && vb == 2) return Kernel<2, 2, true, false>::launch(a, s);
  return cudaErrorInvalidValue;
}

}  // namespace kvq
