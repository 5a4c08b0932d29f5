"""CPU oracle (test infrastructure only; see m3s_oracle's header)."""
