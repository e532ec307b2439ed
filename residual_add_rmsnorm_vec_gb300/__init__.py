"""GB300 (sm_103a) fused residual-add + RMSNorm."""
