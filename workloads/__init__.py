"""Seeded synthetic workloads (input generators and workload table)."""
