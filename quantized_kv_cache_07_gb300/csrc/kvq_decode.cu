// Decode kernels for the symmetric formats (scale only) and bf16 blocks.  The
// kernel template lives in kvq_decode_impl.cuh; the asymmetric formats are
// instantiated in kvq_decode_asym.cu so the two compile in parallel.
#include "kvq_decode_impl.cuh"

namespace kvq {

int decode_ctas_per_sm_for(int k_bits, int v_bits, bool asym, int B) {
  if (asym) return decode_ctas_per_sm_asym(k_bits, v_bits, B);
  if (k_bits == 8 && v_bits == 8) return Kernel<8, 8, false>::ctas_per_sm(B);
  if (k_bits == 4 && v_bits == 4) return Kernel<4, 4, false>::ctas_per_sm(B);
  if (k_bits == 4 && v_bits == 8) return Kernel<4, 8, false>::ctas_per_sm(B);
  if (k_bits == 8 && v_bits == 4) return Kernel<8, 4, false>::ctas_per_sm(B);
  if (k_bits == 16 && v_bits == 16) return Kernel<16, 16, false>::ctas_per_sm(B);
  return 0;
}

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t s) {
  if (a.c.k_offsets) return launch_decode_asym(a, s);
  const int kb = a.c.k_bits, vb = a.c.v_bits;
  if (kb == 8 && vb == 8) return Kernel<8, 8, false>::launch(a, s);
  if (kb == 4 && vb == 4) return Kernel<4, 4, false>::launch(a, s);
  if (kb == 4 && vb == 8) return Kernel<4, 8, false>::launch(a, s);
  if (kb == 8 && vb == 4) return Kernel<8, 4, false>::launch(a, s);
  if (kb == 16 && vb == 16) return Kernel<16, 16, false>::launch(a, s);
  return cudaErrorInvalidValue;
}

}  // namespace kvq
