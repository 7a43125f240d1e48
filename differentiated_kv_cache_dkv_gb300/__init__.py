"""GB300-native DiffKV-style differentiated KV-cache compaction (libdkv)."""
