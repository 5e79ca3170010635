"""GB300-native EAGLE-3 draft-and-verify step: CUDA kernels behind the libeagle3 C ABI.

The compute path is libeagle3.so (hand-written CUDA for sm_103a); this
package only builds it and marshals torch tensors into its C argument
structs.  See include/eagle3.h, include/eagle3_linear.h and include/eagle3_f32.h
for the contract of every entry point.  `tiny` composes the fp32 blocks into the
small lossless configuration (vanilla and speculative greedy decoding).
"""
from ._lib import (EPI_BF16, EPI_BF16_RESIDUAL, EPI_BF16_ROPE, EPI_F32, EPI_SWIGLU, F32_EPI_NONE, F32_EPI_RESIDUAL, F32_EPI_SWIGLU,
                   GREEDY, SAMPLED, TOPK, Eagle3Error, eagle3_accept, eagle3_accept_lazy, eagle3_chain_verify, eagle3_spec_decode_metadata, eagle3_ttt_attn, eagle3_compact_kv, eagle3_draft_tree,
                   eagle3_f32_argmax, eagle3_f32_attn, eagle3_f32_gather, eagle3_f32_linear, eagle3_f32_rmsnorm,
                   eagle3_f32_rope, eagle3_linear, eagle3_rmsnorm, eagle3_verify_attn, eagle3_verify_attn_noalloc,
                   lib)

__all__ = ["GREEDY", "TOPK", "SAMPLED", "Eagle3Error", "eagle3_accept", "eagle3_accept_lazy", "eagle3_chain_verify",
           "eagle3_spec_decode_metadata", "eagle3_ttt_attn", "eagle3_compact_kv", "eagle3_verify_attn",
           "eagle3_verify_attn_noalloc", "eagle3_linear", "eagle3_draft_tree", "eagle3_rmsnorm", "EPI_BF16", "EPI_F32",
           "EPI_BF16_RESIDUAL", "EPI_BF16_ROPE", "EPI_SWIGLU", "F32_EPI_NONE", "F32_EPI_RESIDUAL", "F32_EPI_SWIGLU",
           "eagle3_f32_linear", "eagle3_f32_rmsnorm", "eagle3_f32_rope", "eagle3_f32_gather", "eagle3_f32_argmax",
           "eagle3_f32_attn", "lib"]
