"""GB300-native batched lossless speculative verification (binding filled in below)."""
