"""GB300-native residue-compensated block-scaled FP4 linear layers."""
