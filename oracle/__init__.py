"""CPU oracle of the AWQ calibration hot path (test infrastructure only)."""
