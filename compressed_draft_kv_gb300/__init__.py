"""GB300-native MASW draft memory and attention (C-ABI library + thin binding)."""
