"""GB300-native segmented gather LoRA apply (SGMV shrink / expand / fused apply)."""
