"""Paged decode/verify attention and speculative acceptance for GB300."""
