"""B300-native selective state-space scan (Mamba-1 diagonal form and Mamba-2 SSD form)."""
