"""GB300 (sm_103a) exact attention: FlashAttention forward and backward."""
