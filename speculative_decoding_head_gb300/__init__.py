"""GB300-native DSpark round: Markov-head draft tail, confidence-scheduled planner, lossless ragged verify."""
