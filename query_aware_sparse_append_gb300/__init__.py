"""Query-aware sparse paged decode attention for GB300 (sm_103a)."""
