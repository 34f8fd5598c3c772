// Select kernel: one CTA of kSelThreads per (layer, sequence); the work is
// select_group (select_body.cuh).
#include "select_body.cuh"

namespace confkv {

template <int D, bool kSmemKeys, bool kDevStep, bool kOrdered>
__global__ void __launch_bounds__(kSelThreads, 4) select_kernel(Shape s, Dev d, long long step_arg,
                                                             int32_t* __restrict__ evicted_out,
                                                             int32_t* __restrict__ nevict_out,
                                                             SelSmem sm) {
  extern __shared__ __align__(16) unsigned char dsm[];
  __shared__ SelShared sh;
  pdl_wait();
  select_group<D, kSmemKeys, kDevStep, kOrdered, kSelThreads, true>(s, d, step_arg, blockIdx.x, evicted_out,
                                                                    nevict_out, sm, dsm, sh);
}

template <int D, bool kSmemKeys, bool kDevStep, bool kOrdered>
static int launch_select_t(const Shape& s, const Dev& d, long long step, int32_t* evicted_pos,
                           int32_t* n_evicted, const SelSmem& p, cudaStream_t stream) {
  static int configured[kMaxDevices] = {};
  if (p.bytes > 48 * 1024 &&
      ensure_smem(select_kernel<D, kSmemKeys, kDevStep, kOrdered>, p.bytes, configured) != cudaSuccess)
    return -1;
  return launch_pdl(select_kernel<D, kSmemKeys, kDevStep, kOrdered>, dim3(s.L * s.B), dim3(kSelThreads),
                    (size_t)p.bytes, stream, s, d, step, evicted_pos, n_evicted, p) == cudaSuccess
             ? 0
             : -1;
}

template <int D, bool kSmemKeys, bool kDevStep>
static int launch_select_o(const Shape& s, const Dev& d, long long step, int32_t* evicted_pos,
                           int32_t* n_evicted, const SelSmem& p, cudaStream_t stream) {
  return s.compaction == 1
             ? launch_select_t<D, kSmemKeys, kDevStep, true>(s, d, step, evicted_pos, n_evicted, p, stream)
             : launch_select_t<D, kSmemKeys, kDevStep, false>(s, d, step, evicted_pos, n_evicted, p, stream);
}

template <int D, bool kSmemKeys>
static int launch_select_s(const Shape& s, const Dev& d, long long step, int32_t* evicted_pos,
                           int32_t* n_evicted, const SelSmem& p, cudaStream_t stream) {
  return step >= 0 ? launch_select_o<D, kSmemKeys, false>(s, d, step, evicted_pos, n_evicted, p, stream)
                   : launch_select_o<D, kSmemKeys, true>(s, d, step, evicted_pos, n_evicted, p, stream);
}

int launch_select(const Shape& s, const Dev& d, long long step, int32_t* evicted_pos,
                  int32_t* n_evicted, cudaStream_t stream) {
  const SelSmem p = plan_select(s);
  const bool smem_keys = p.off_key >= 0;
  if (s.D == 128)
    return smem_keys ? launch_select_s<128, true>(s, d, step, evicted_pos, n_evicted, p, stream)
                     : launch_select_s<128, false>(s, d, step, evicted_pos, n_evicted, p, stream);
  return smem_keys ? launch_select_s<64, true>(s, d, step, evicted_pos, n_evicted, p, stream)
                   : launch_select_s<64, false>(s, d, step, evicted_pos, n_evicted, p, stream);
}

}  // namespace confkv
