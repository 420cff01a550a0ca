// k_tc64.cu -- the state-form tensor-core forward at head dimension 64: the kernels of
// tc_state_form.cuh instantiated with 64-wide operand tiles (8 KB state images, N = 64
// cached-read MMAs, K = 64 contractions over the head dimension), in a translation unit
// of their own so that both widths compile in parallel.
#include "tc_state_form.cuh"

namespace mc {

cudaError_t launch_forward_tc64(const Problem &p, const FwdArgs &fa, void *scratch, cudaStream_t s)
{
    return forward_impl<64>(p, fa, scratch, s);
}

cudaError_t launch_state_tc_segments64(const Problem &p, const FwdArgs &fa, const TcSegTables &tb, void *scratch,
                                       cudaStream_t s)
{
    return state_segments_impl<64>(p, fa, tb, scratch, s);
}

cudaError_t launch_readout_tc_segments64(const Problem &p, const FwdArgs &fa, const TcSegTables &tb, void *scratch,
                                         cudaStream_t s)
{
    return readout_segments_impl<64>(p, fa, tb, scratch, s);
}

cudaError_t take_tc64_abort(int *was_set) { return take_tc_abort(was_set); }

}  // namespace mc
