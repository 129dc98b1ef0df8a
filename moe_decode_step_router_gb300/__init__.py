"""GB300-native small-M MoE decode/verify step (binding is in `moestep`)."""
