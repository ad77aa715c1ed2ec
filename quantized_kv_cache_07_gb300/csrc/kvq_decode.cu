// Decode kernels for the symmetric formats (scale only) and bf16 blocks with
// the fp16 or int8 query.  The kernel template lives in kvq_decode_impl.cuh;
// the asymmetric formats (kvq_decode_asym.cu) and the two-part fp16 query
// (kvq_decode_q32.cu) are instantiated in their own translation units so the
// three compile in parallel.
#include "kvq_decode_impl.cuh"

namespace kvq {

int decode_ctas_per_sm_for(int k_bits, int v_bits, bool asym, int q_bits, int B, bool rows) {
  if (q_bits == 32 && k_bits != 16) return decode_ctas_per_sm_q32(k_bits, v_bits, asym, B, rows);
  if (asym) return decode_ctas_per_sm_asym(k_bits, v_bits, B, rows);
  if (k_bits == 8 && v_bits == 8) return Kernel<8, 8, false, false>::ctas_per_sm(B, rows);
  if (k_bits == 4 && v_bits == 4) return Kernel<4, 4, false, false>::ctas_per_sm(B, rows);
  if (k_bits == 4 && v_bits == 8) return Kernel<4, 8, false, false>::ctas_per_sm(B, rows);
  if (k_bits == 8 && v_bits == 4) return Kernel<8, 4, false, false>::ctas_per_sm(B, rows);
  if (k_bits == 2 && v_bits == 2) return Kernel<2, 2, false, false>::ctas_per_sm(B, rows);
  if (k_bits == 16 && v_bits == 16) return Kernel<16, 16, false, false>::ctas_per_sm(B, rows);
  return 0;
}

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t s) {
  const int kb = a.c.k_bits, vb = a.c.v_bits;
  if (a.c.q_bits == 32 && kb != 16) return launch_decode_q32(a, s);
  if (a.c.asym) return launch_decode_asym(a, s);
  if (kb == 8 && vb == 8) return Kernel<8, 8, false, false>::launch(a, s);
  if (kb == 4 && vb == 4) return Kernel<4, 4, false, false>::launch(a, s);
  if (kb == 4 && vb == 8) return Kernel<4, 8, false, false>::launch(a, s);
  if (kb == 8 && vb == 4) return Kernel<8, 4, false, false>::launch(a, s);
  if (kb == 2 && vb == 2) return Kernel<2, 2, false, false>::launch(a, s);
  if (kb == 16 && vb == 16) return Kernel<16, 16, false, false>::launch(a, s);
  return cudaErrorInvalidValue;
}

}  // namespace kvq
