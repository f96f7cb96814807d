"""CPU oracle of the EAGLE-3 drafter draft round (test infrastructure only)."""
