"""paged_kv_cache_101_gb300: placeholder until the binding lands."""
