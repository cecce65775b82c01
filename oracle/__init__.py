"""CPU oracle for blended prefill: test infrastructure only (see blend_oracle.py)."""
