"""GB300-native DSpark sequential Markov draft-sampling loop."""
