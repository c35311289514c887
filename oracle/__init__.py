"""CPU float64 oracle (test infrastructure only; see dflash2_oracle's header)."""
