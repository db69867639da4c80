"""GB300 (sm_103a) single-token grouped-query decode attention."""
