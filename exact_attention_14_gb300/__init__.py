"""GB300 exact attention: fused forward and split-KV decode (binding filled in below)."""
