// bf16 V-cache instantiations of the AV kernel.
#include "gqa_av_instances.cuh"
namespace gqa_av {
GQA_AV_INSTANTIATE_ALL(Bf16Tag)
}  // namespace gqa_av
