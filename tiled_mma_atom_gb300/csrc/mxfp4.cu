// mxfp4.cu — placeholder until the block-scaled tcgen05 kernel lands.
#include "internal.h"

namespace tmg {

cudaError_t launch_mxfp4(const Mxfp4Args &a, int num_sms, const ErrCtx &err, cudaStream_t s)
{
    (void)a;
    (void)num_sms;
    (void)err;
    (void)s;
    return cudaErrorNotSupported;
}

}  // namespace tmg
