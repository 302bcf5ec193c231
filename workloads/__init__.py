"""Seeded synthetic workloads and input generators (no attention arithmetic here)."""
