"""The fp64 CPU oracle of the attention step (test infrastructure; see attention.py's header)."""
