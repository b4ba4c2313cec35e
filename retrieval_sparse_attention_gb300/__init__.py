"""GCA hot path on GB300 (sm_103a)."""
