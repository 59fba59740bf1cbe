"""GB300-native fused data-parallel step: bucketed gradient reduction,
AdamW and parameter redistribution in one pass (placeholder; the binding
arrives with the C-ABI library)."""
