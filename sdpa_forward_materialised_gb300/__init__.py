"""GB300 (sm_103a) materialised-probability SDPA forward: (O, P)."""
