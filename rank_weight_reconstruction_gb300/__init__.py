"""Theta-bundle reconstruction linear for GB300 (sm_103a)."""
