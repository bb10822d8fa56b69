"""GB300-native Mamba-2 SSD hot path (binding filled in below)."""
