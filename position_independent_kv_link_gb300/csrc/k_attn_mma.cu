// Tensor-core paged attention (bf16, head_dim 128): placeholder routing to the generic kernel.
#include "pic_internal.h"

namespace pic {
void launch_attention_simt(const AttnArgs& a, cudaStream_t st);
void launch_attention_mma(const AttnArgs& a, cudaStream_t st) { launch_attention_simt(a, st); }
}  // namespace pic
