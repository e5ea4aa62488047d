"""CPU oracle (test infrastructure only; see indexer_topk.py)."""
