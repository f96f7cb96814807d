"""EAGLE-3 drafter draft round for greedy speculative decoding on GB300 (sm_103a)."""
