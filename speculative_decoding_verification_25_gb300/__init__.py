"""Batched speculative-decoding verify-and-accept on GB300 (sm_103a)."""
