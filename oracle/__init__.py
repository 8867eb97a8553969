"""Oracle package: test infrastructure only (see moe_oracle.py)."""
