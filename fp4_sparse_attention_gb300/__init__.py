"""GB300-native FP4 lightning-indexer scorer.

The scorer computes ``logits[t, s] = sum_h w[t, h] * ReLU(q[t, h] . k[s])`` over
a paged FP4 K cache (E2M1 codes with MXFP4 or NVFP4 block scales), masks the
positions a row cannot see to -inf, and returns the full logits, a per-128-key
block max of the unweighted scores, or the top-k positions of each row.

All arithmetic runs in the CUDA library ``libfp4idx.so`` (C ABI in
``include/fp4idx.h``); :mod:`fp4_sparse_attention_gb300.binding` marshals
torch device tensors into it.  There is no CPU fallback: the ops raise if the
library is missing.
"""

MXFP4 = 0
NVFP4 = 1

__all__ = ["MXFP4", "NVFP4"]
