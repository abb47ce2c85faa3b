"""CPU fp64 oracle (test infrastructure only; see ``thd_oracle``)."""
