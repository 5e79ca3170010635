"""GB300-native EAGLE-3 draft-and-verify step: CUDA kernels behind the libeagle3 C ABI.

The compute path is libeagle3.so (hand-written CUDA for sm_103a); this
package only builds it and marshals torch tensors into its C argument
structs.  See include/eagle3.h for the contract of every entry point.
"""
from ._lib import (EPI_BF16, EPI_BF16_RESIDUAL, EPI_F32, EPI_SWIGLU, GREEDY, SAMPLED, TOPK, Eagle3Error,
                   eagle3_accept, eagle3_compact_kv, eagle3_draft_tree, eagle3_linear, eagle3_rmsnorm,
                   eagle3_verify_attn, lib)

__all__ = ["GREEDY", "TOPK", "SAMPLED", "Eagle3Error", "eagle3_accept", "eagle3_compact_kv",
           "eagle3_verify_attn", "eagle3_linear", "eagle3_draft_tree", "eagle3_rmsnorm", "EPI_BF16", "EPI_F32", "EPI_BF16_RESIDUAL", "EPI_SWIGLU", "lib"]
