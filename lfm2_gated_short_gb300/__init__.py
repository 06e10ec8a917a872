"""LFM2 gated short convolution (ShortConv) on GB300 (sm_103a)."""
